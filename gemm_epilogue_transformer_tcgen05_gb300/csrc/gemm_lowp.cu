// tf32 (fp32 operands) and e4m3 GEMM-epilogue variants (K-major operands).
#include "coda_internal.h"

namespace coda {
const VariantEntry g_variants_lowp[] = {
    CODA_VARIANT(KIND_TF32, EPI_STORE, false, false, DT_F32, DT_F32, false),
    CODA_VARIANT(KIND_TF32, EPI_RESID, false, false, DT_F32, DT_F32, false),
    CODA_VARIANT(KIND_TF32, EPI_ROWSCALE, false, false, DT_F32, DT_F32, false),
    CODA_VARIANT(KIND_E4M3, EPI_SWIGLU, false, false, DT_E4M3, DT_BF16, false),
    CODA_VARIANT(KIND_E4M3, EPI_RESID, false, false, DT_BF16, DT_BF16, false),
    CODA_VARIANT(KIND_E4M3, EPI_STORE, false, false, DT_BF16, DT_BF16, false),
};
const int g_num_variants_lowp = sizeof(g_variants_lowp) / sizeof(g_variants_lowp[0]);
}  // namespace coda
