// e4m3 variants of the FP8 MLP's training path: the forward that also saves Z = [G | U],
// and the backward GEMMs (MN-major operands where the backward reads a tensor transposed).
#include "coda_internal.h"

namespace coda {
const VariantEntry g_variants_fp8[] = {
    CODA_VARIANT(KIND_E4M3, EPI_SWIGLU, false, false, DT_E4M3, DT_BF16, true),
    CODA_VARIANT(KIND_E4M3, EPI_SWIGLU_BWD, false, true, DT_E4M3, DT_BF16, false),
    CODA_VARIANT(KIND_E4M3, EPI_RMSBWD, false, true, DT_BF16, DT_BF16, false),
    CODA_VARIANT(KIND_E4M3, EPI_STORE, true, true, DT_F32, DT_BF16, false),
};
const int g_num_variants_fp8 = sizeof(g_variants_fp8) / sizeof(g_variants_fp8[0]);
}  // namespace coda
