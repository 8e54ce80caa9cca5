// Backward-chain GEMM-epilogue variants (bf16; MN-major operands for dX and dW GEMMs).
#include "coda_internal.h"

namespace coda {
const VariantEntry g_variants_bwd[] = {
    CODA_VARIANT(KIND_BF16, EPI_SWIGLU_BWD, false, true, DT_BF16, DT_BF16, false),
    CODA_VARIANT(KIND_BF16, EPI_RMSBWD, false, true, DT_BF16, DT_BF16, false),
    CODA_VARIANT(KIND_BF16, EPI_STORE, false, true, DT_BF16, DT_BF16, false),
    CODA_VARIANT(KIND_BF16, EPI_STORE, true, true, DT_F32, DT_BF16, false),
    CODA_VARIANT(KIND_BF16, EPI_STORE, true, false, DT_BF16, DT_BF16, false),
};
const int g_num_variants_bwd = sizeof(g_variants_bwd) / sizeof(g_variants_bwd[0]);
}  // namespace coda
