// NVFP4 variants: block-scaled e2m1 operands (CTA pairs, MMA N = 256, one accumulator): the plain GEMM, the
// residual program of a down projection, the SwiGLU program with an NVFP4 or bf16 output, and for the
// backward the RMSNorm-backward program (bf16 output, bf16 side inputs).  The SwiGLU backward, whose
// epilogue moves as many bytes as its short mainloop takes time (Z read, e written), uses MMA N = 128 and
// two accumulators, so that each tile's epilogue runs under the next tile's MMAs.
#include "coda_internal.h"

namespace coda {
const VariantEntry g_variants_fp4[] = {
    CODA_VARIANT_FP4(EPI_STORE, DT_F32),
    CODA_VARIANT_FP4(EPI_STORE, DT_BF16),
    CODA_VARIANT_FP4(EPI_RESID, DT_BF16),
    CODA_VARIANT_FP4(EPI_SWIGLU, DT_E2M1),
    CODA_VARIANT_FP4(EPI_SWIGLU, DT_BF16),
    CODA_VARIANT_FP4_N(EPI_SWIGLU_BWD, DT_BF16, 128),
    CODA_VARIANT_FP4(EPI_RMSBWD, DT_BF16),
};
const int g_num_variants_fp4 = sizeof(g_variants_fp4) / sizeof(g_variants_fp4[0]);
}  // namespace coda
