// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once
#include <atomic>

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "coda_gemm.cuh"

namespace coda {

// One compiled GEMM-epilogue variant.
struct VariantKey {
  int kind, epi, a_mn, b_mn, out_dt, side_dt, aux;
};
struct VariantEntry {
  VariantKey key;
  GemmLaunchFn fn;
  int smem_bytes;
  int stages;
  int cg;          // CTAs per MMA group (2 = CTA pair)
  int un;          // MMA N (B rows per tile)
  int bn_out;      // output columns per tile
  int b_box;       // B rows per TMA copy
  int bk;          // K elements per pipeline stage
  int ow;          // chunks of 32 output columns per TMA store (box width of the output maps)
};

// Tables defined by the instantiation units.
extern const VariantEntry g_variants_fwd[];
extern const int g_num_variants_fwd;
extern const VariantEntry g_variants_bwd[];
extern const int g_num_variants_bwd;
extern const VariantEntry g_variants_lowp[];
extern const int g_num_variants_lowp;
extern const VariantEntry g_variants_fp8[];
extern const int g_num_variants_fp8;
extern const VariantEntry g_variants_fp4[];
extern const int g_num_variants_fp4;

const VariantEntry* find_variant(const VariantKey& k);

// 1 (default): kernels are launched with a programmatic dependency on the previous kernel of the
// stream (their launch overlaps its tail); 0: plain stream serialisation.
extern std::atomic<int> g_launch_overlap;

// Small bandwidth-bound kernels (coda_small.cu).  Arguments are validated by the caller.
// launch_row_rms: `zero` (optional) is a float the kernel sets to 0 before its dependants run;
// `beside`: one CTA per SM, leaving room for the next GEMM's CTA (a chain whose GEMM reads r
// only in its epilogue); otherwise the many-CTA pass.
cudaError_t launch_partial_reduce(const float* partials, int64_t ld, int nparts, int64_t M, float inv_d, float eps,
                                  int mode, const float* rowscale, float* out, cudaStream_t s);
cudaError_t launch_row_rms(const void* X, int64_t M, int64_t d, int64_t ld, float eps, float* r, cudaStream_t s,
                           int sms, float* zero = nullptr, bool beside = false);
cudaError_t launch_col_reduce(const float* parts, int64_t nblocks, int64_t N, int64_t ld, float* out,
                              cudaStream_t s);
enum FoldOut { FOLD_OUT_BF16 = 0, FOLD_OUT_F32 = 1, FOLD_OUT_E4M3 = 2 };
cudaError_t launch_fold_gain(const void* W, int64_t N, int64_t K, int64_t ld_in, const float* g, float inv_scale,
                             void* W_out, int64_t ld_out, int out_kind, cudaStream_t s, int sms);
cudaError_t launch_rope_table(int seq_len, int head_dim, double base, float* cos_out, float* sin_out,
                              cudaStream_t s);
cudaError_t launch_rms_gain(const void* X, int64_t M, int64_t d, int64_t ld, const float* g, float eps, float* r,
                            void* U, int64_t ldu, cudaStream_t s);
cudaError_t launch_rope_bwd(const void* dout, const void* out, int64_t M, int64_t N, int64_t ld, const float* r,
                            const float* cs, const float* sn, int seq_len, int head_dim, int rope_ncols, int64_t H,
                            void* e, int64_t lde, float* c, cudaStream_t s);
cudaError_t launch_quantize_e4m3(const void* X, int64_t M, int64_t N, int64_t ldx, float inv_scale, void* Q,
                                 int64_t ldq, float* amax, cudaStream_t s, int sms);
cudaError_t launch_quantize_nvfp4(const void* X, int64_t R, int64_t K, int64_t ldx, float s, void* Q, int64_t ldq_bytes,
                                  uint8_t* sf, float* amax, cudaStream_t st, int sms);
cudaError_t launch_quantize_nvfp4_t(const void* X, int64_t R, int64_t C, int64_t ldx, bool swiglu, float s, void* Q,
                                    int64_t ldq_bytes, uint8_t* sf, void* Qr, int64_t ldqr_bytes, uint8_t* sfr,
                                    float* amax, cudaStream_t st, int sms);
cudaError_t launch_xent_reduce(const float* Pm, const float* Ps, int64_t ld, int nparts, int64_t M, const float* T,
                               const int* targets, int64_t V, float* lse, float* loss, float* mean, cudaStream_t s);

}  // namespace coda

namespace coda {
template <class C>
constexpr VariantEntry make_variant(VariantKey k) {
  return {k, &launch_gemm<C>, C::SMEM_BYTES, C::STAGES, C::CG, C::UN, C::BN_OUT, C::B_BOX, C::BK, C::OW};
}
}  // namespace coda
#define CODA_VARIANT(KIND, EPI, AMN, BMN, OUT, SIDE, AUX) \
  make_variant<GemmCfg<KIND, EPI, AMN, BMN, OUT, SIDE, AUX>>(VariantKey{KIND, EPI, AMN, BMN, OUT, SIDE, AUX})
// NVFP4 variants: CTA pairs with MMA N = 256 and one accumulator, or MMA N = 128 and two
#define CODA_VARIANT_FP4_N(EPI, OUT, UN_)                                                 \
  make_variant<GemmCfg<KIND_NVFP4, EPI, false, false, OUT, DT_BF16, false, 2, UN_>>( \
      VariantKey{KIND_NVFP4, EPI, false, false, OUT, DT_BF16, false})
#define CODA_VARIANT_FP4(EPI, OUT) CODA_VARIANT_FP4_N(EPI, OUT, 256)
