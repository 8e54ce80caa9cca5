// Forward-chain GEMM-epilogue variants (bf16, both operands K-major).
#include "coda_internal.h"

namespace coda {
const VariantEntry g_variants_fwd[] = {
    CODA_VARIANT(KIND_BF16, EPI_STORE, false, false, DT_BF16, DT_BF16, false),
    CODA_VARIANT(KIND_BF16, EPI_STORE, false, false, DT_F32, DT_BF16, false),
    CODA_VARIANT(KIND_BF16, EPI_RESID, false, false, DT_BF16, DT_BF16, false),
    CODA_VARIANT(KIND_BF16, EPI_RESID, false, false, DT_BF16, DT_BF16, true),
    CODA_VARIANT(KIND_BF16, EPI_ROWSCALE, false, false, DT_BF16, DT_BF16, false),
    CODA_VARIANT(KIND_BF16, EPI_SWIGLU, false, false, DT_BF16, DT_BF16, false),
    CODA_VARIANT(KIND_BF16, EPI_SWIGLU, false, false, DT_BF16, DT_BF16, true),
    CODA_VARIANT(KIND_BF16, EPI_ROPE, false, false, DT_BF16, DT_BF16, false),
    CODA_VARIANT(KIND_BF16, EPI_XENT, false, false, DT_BF16, DT_BF16, false),
    CODA_VARIANT(KIND_BF16, EPI_XENT_BWD, false, false, DT_BF16, DT_BF16, false),
};
const int g_num_variants_fwd = sizeof(g_variants_fwd) / sizeof(g_variants_fwd[0]);
}  // namespace coda
