// Bandwidth- and latency-bound helper kernels of the GEMM-epilogue chains:
//   * the light row reduce that turns per-tile partial sums into the RMS scale r (or the
//     backward coefficient c) — "CODA: new research optimizes Transformer training with
//     GEMM-epilogue programming" (kucoin.com news flash), section "El epílogo esconde un
//     tesoro": partial RMS from the first GEMM, combined by a very light reduce kernel;
//   * a full-row RMS scale (one pass over an activation) for chains that start from a
//     stored activation;
//   * the column reduce of per-block column partials (RMSNorm gain gradient);
//   * the gain fold W' = W diag(g) (weight preparation for the deferred-r GEMM);
//   * the RoPE cos/sin table;
//   * e4m3 and NVFP4 quantisers.
#include <cuda_bf16.h>

#include <type_traits>

#include "coda_internal.h"

namespace coda {

// Launch with a programmatic dependency on the previous kernel of the stream (when enabled):
// every kernel here first waits (griddepcontrol.wait) for that kernel's completion, then lets
// the next kernel launch; only the launch latency overlaps the previous kernel's tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), unsigned grid, unsigned block, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = g_launch_overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------- partial reduce
// Partials stored [nparts, M], so a warp's load of 32 consecutive rows is coalesced.
// Few parts (the chains' own, e.g. 8 for a 2048-wide layer): one thread per row, four running
// sums (part t into sum t % 4) added as (s0 + s1) + (s2 + s3).  The kernel uses no shared
// memory, so the next GEMM's CTA (all but a few KB of an SM's shared memory) can start beside
// it (the block forward ran 0.2% slower with the shared-merge kernel below in its place).
// Many parts (the LM head's 501): a CTA takes 32 rows and splits the parts over its 8 warps,
// warp w adding parts w, w + 8, ... in order (four loads in flight), and the warps' sums are
// added as ((w0 + w4) + (w1 + w5)) + ((w2 + w6) + (w3 + w7)).  One thread per row over all
// parts ran at 1.3 TB/s there (64 CTAs for 16384 rows).
__device__ __forceinline__ float reduce_finish(float tot, int mode, float inv_d, float eps, float rs) {
  return mode == 0 ? rsqrtf(fmaf(tot, inv_d, eps)) : rs * (tot * inv_d);
}
__global__ void partial_reduce_kernel(const float* __restrict__ P, int64_t ld, int nparts, int64_t M, float inv_d,
                                      float eps, int mode, const float* __restrict__ rowscale,
                                      float* __restrict__ out) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= M) return;
  float s4[4] = {0.f, 0.f, 0.f, 0.f};
  int t = 0;
  for (; t + 4 <= nparts; t += 4) {
#pragma unroll
    for (int k = 0; k < 4; ++k) s4[k] += __ldg(P + (int64_t)(t + k) * ld + i);
  }
  for (; t < nparts; ++t) s4[0] += __ldg(P + (int64_t)t * ld + i);
  out[i] = reduce_finish((s4[0] + s4[1]) + (s4[2] + s4[3]), mode, inv_d, eps, mode ? __ldg(rowscale + i) : 0.f);
}
constexpr int PR_WARPS = 8;
__global__ void __launch_bounds__(32 * PR_WARPS)
    partial_reduce_split_kernel(const float* __restrict__ P, int64_t ld, int nparts, int64_t M, float inv_d,
                                float eps, int mode, const float* __restrict__ rowscale, float* __restrict__ out) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  __shared__ float st[PR_WARPS][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t i = (int64_t)blockIdx.x * 32 + lane;
  float s = 0.f;
  if (i < M) {
    int t = w;
    for (; t + 3 * PR_WARPS < nparts; t += 4 * PR_WARPS) {
      float v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = __ldg(P + (int64_t)(t + k * PR_WARPS) * ld + i);
#pragma unroll
      for (int k = 0; k < 4; ++k) s += v[k];
    }
    for (; t < nparts; t += PR_WARPS) s += __ldg(P + (int64_t)t * ld + i);
  }
  st[w][lane] = s;
  __syncthreads();
  if (w == 0 && i < M) {
    const float tot = ((st[0][lane] + st[4][lane]) + (st[1][lane] + st[5][lane])) +
                      ((st[2][lane] + st[6][lane]) + (st[3][lane] + st[7][lane]));
    out[i] = reduce_finish(tot, mode, inv_d, eps, mode ? __ldg(rowscale + i) : 0.f);
  }
}

cudaError_t launch_partial_reduce(const float* partials, int64_t ld, int nparts, int64_t M, float inv_d, float eps,
                                  int mode, const float* rowscale, float* out, cudaStream_t s) {
  if (nparts <= 16) {
    const int threads = 256;
    launch_k(partial_reduce_kernel, (unsigned)((M + threads - 1) / threads), threads, s, partials, ld, nparts, M, inv_d,
             eps, mode, rowscale, out);
  } else {
    launch_k(partial_reduce_split_kernel, (unsigned)((M + 31) / 32), 32 * PR_WARPS, s, partials, ld, nparts, M, inv_d,
             eps, mode, rowscale, out);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------- full-row RMS
// Sum of squares of R rows of bf16 (nvec 16-byte chunks each, 8 values a chunk) across one
// warp, in the order both row-RMS kernels share, so they give the same bits: lane l takes
// chunks l + 32 j; in the main loop chunk v + 32 k goes into running sum k (four loads in
// flight a row), in the tail into sum 0; then (s0 + s1) + (s2 + s3) and the lanes by xor
// shuffles.  The R rows' loads are issued together.
template <int R>
__device__ __forceinline__ void rows_sumsq(const uint4* const (&src)[R], int64_t nvec, int lane, float (&out)[R]) {
  float acc[R][4];
#pragma unroll
  for (int j = 0; j < R; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  int64_t v = lane;
  for (; v + 96 < nvec; v += 128) {
    uint4 u[R][4];
#pragma unroll
    for (int j = 0; j < R; ++j)
#pragma unroll
      for (int k = 0; k < 4; ++k) u[j][k] = __ldcs(src[j] + v + 32 * k);
#pragma unroll
    for (int j = 0; j < R; ++j)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t w[4] = {u[j][k].x, u[j][k].y, u[j][k].z, u[j][k].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xFFFF0000u);
          acc[j][k] = fmaf(lo, lo, fmaf(hi, hi, acc[j][k]));
        }
      }
  }
  for (; v < nvec; v += 32) {
    uint4 u[R];
#pragma unroll
    for (int j = 0; j < R; ++j) u[j] = __ldcs(src[j] + v);
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const uint32_t w[4] = {u[j].x, u[j].y, u[j].z, u[j].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xFFFF0000u);
        acc[j][0] = fmaf(lo, lo, fmaf(hi, hi, acc[j][0]));
      }
    }
  }
#pragma unroll
  for (int j = 0; j < R; ++j) {
    float s = (acc[j][0] + acc[j][1]) + (acc[j][2] + acc[j][3]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    out[j] = s;
  }
}

// One warp per row, many CTAs: the fastest pass on its own.
__global__ void row_rms_kernel(const __nv_bfloat16* __restrict__ X, int64_t M, int64_t d, int64_t ld, float eps,
                               float* __restrict__ r, float* __restrict__ zero) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  // a chain's amax accumulator, reset here rather than by a separate memset: the next kernel
  // of the stream reads it only after this one has completed
  if (zero && blockIdx.x == 0 && threadIdx.x == 0) *zero = 0.f;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= M) return;
  const uint4* const src[1] = {reinterpret_cast<const uint4*>(X + row * ld)};
  float s[1];
  rows_sumsq<1>(src, d >> 3, lane, s);
  if (lane == 0) r[row] = rsqrtf(fmaf(s[0], 1.0f / (float)d, eps));
}

// One CTA of 8 warps per SM, a warp taking 4 rows at a time (16 loads in flight a lane), at most
// 128 registers a thread: the GEMM that follows in a chain (6 warps of up to 128 registers, up
// to 226 KB of shared memory) fits on the SM beside it, so a GEMM that reads r only in its
// epilogue runs its first mainloop under this pass.  On its own the pass is slower than the
// many-CTA kernel (16384 x 8192: 55 against 37 us; each warp's groups are serial DRAM round
// trips, and prefetching the next group into L2 did not help), so only the chains use it.
constexpr int RR_WARPS = 8, RR_ROWS = 4;
__global__ void __launch_bounds__(32 * RR_WARPS, 2)
    row_rms_beside_kernel(const __nv_bfloat16* __restrict__ X, int64_t M, int64_t d, int64_t ld, float eps,
                          float* __restrict__ r, float* __restrict__ zero) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  if (zero && blockIdx.x == 0 && threadIdx.x == 0) *zero = 0.f;
  const int lane = threadIdx.x & 31;
  const int64_t step = (int64_t)gridDim.x * RR_WARPS;
  for (int64_t grp = (int64_t)blockIdx.x * RR_WARPS + (threadIdx.x >> 5); grp * RR_ROWS < M; grp += step) {
    const int64_t row0 = grp * RR_ROWS;
    const uint4* src[RR_ROWS];
#pragma unroll
    for (int j = 0; j < RR_ROWS; ++j)   // rows past M re-read row0 (always in range) and are not stored
      src[j] = reinterpret_cast<const uint4*>(X + (row0 + j < M ? row0 + j : row0) * ld);
    float s[RR_ROWS];
    rows_sumsq<RR_ROWS>(src, d >> 3, lane, s);
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < RR_ROWS; ++j)
        if (row0 + j < M) r[row0 + j] = rsqrtf(fmaf(s[j], 1.0f / (float)d, eps));
    }
  }
}

cudaError_t launch_row_rms(const void* X, int64_t M, int64_t d, int64_t ld, float eps, float* r, cudaStream_t s,
                           int sms, float* zero, bool beside) {
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(X);
  if (beside) {
    // the carve-out the GEMM beside it needs; set once (a function-local static is initialised once)
    static const cudaError_t attr = cudaFuncSetAttribute(
        row_rms_beside_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (attr != cudaSuccess) return attr;
    const int64_t groups = (M + RR_ROWS - 1) / RR_ROWS;
    const int64_t need = (groups + RR_WARPS - 1) / RR_WARPS;
    const unsigned grid = (unsigned)(need < sms ? need : sms);
    launch_k(row_rms_beside_kernel, grid, 32 * RR_WARPS, s, x, M, d, ld, eps, r, zero);
  } else {
    const int rows_per_block = 8;
    const int64_t blocks = (M + rows_per_block - 1) / rows_per_block;
    launch_k(row_rms_kernel, (unsigned)blocks, 32 * rows_per_block, s, x, M, d, ld, eps, r, zero);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------- RMS + gain broadcast
// One warp per row: r = 1 / sqrt(mean x^2 + eps) and u = x * g (bf16), one pass over X.
__global__ void rms_gain_kernel(const __nv_bfloat16* __restrict__ X, int64_t M, int64_t d, int64_t ld,
                                const float* __restrict__ g, float eps, float* __restrict__ r,
                                __nv_bfloat16* __restrict__ U, int64_t ldu) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= M) return;
  const uint4* src = reinterpret_cast<const uint4*>(X + row * ld);
  uint4* dst = reinterpret_cast<uint4*>(U + row * ldu);
  const int64_t nvec = d >> 3;
  float acc = 0.f;
  for (int64_t v = lane; v < nvec; v += 32) {
    const uint4 u = __ldcs(src + v);
    const float4 g0 = __ldg(reinterpret_cast<const float4*>(g + 8 * v));
    const float4 g1 = __ldg(reinterpret_cast<const float4*>(g + 8 * v + 4));
    const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xFFFF0000u);
      acc = fmaf(lo, lo, fmaf(hi, hi, acc));
      __nv_bfloat162 b = __floats2bfloat162_rn(lo * gv[2 * e], hi * gv[2 * e + 1]);
      o[e] = *reinterpret_cast<uint32_t*>(&b);
    }
    dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) r[row] = rsqrtf(fmaf(acc, 1.0f / (float)d, eps));
}

cudaError_t launch_rms_gain(const void* X, int64_t M, int64_t d, int64_t ld, const float* g, float eps, float* r,
                            void* U, int64_t ldu, cudaStream_t s) {
  const int rows_per_block = 8;
  const int64_t blocks = (M + rows_per_block - 1) / rows_per_block;
  launch_k(rms_gain_kernel, (unsigned)blocks, 32 * rows_per_block, s, static_cast<const __nv_bfloat16*>(X), M, d, ld,
                                                                    g, eps, r, static_cast<__nv_bfloat16*>(U), ldu);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- RoPE backward
// One warp per row: e = r * R(-phi) dout (the transpose of the forward rotation on the
// first rope_ncols columns, plain copy after), and c = r * s / H with
// s = r * sum_n dout_n out_n (= sum_n e_n Z_n, the rotation keeps inner products).
__global__ void rope_bwd_kernel(const __nv_bfloat16* __restrict__ dout, const __nv_bfloat16* __restrict__ out,
                                int64_t M, int64_t N, int64_t ld, const float* __restrict__ r,
                                const float* __restrict__ cs, const float* __restrict__ sn, int seq_len, int head_dim,
                                int rope_ncols, float inv_h, __nv_bfloat16* __restrict__ e, int64_t lde,
                                float* __restrict__ c) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= M) return;
  const float rr = __ldg(r + row);
  const int pos = (int)(row % seq_len);
  const int half = head_dim >> 1;
  const uint4* dsrc = reinterpret_cast<const uint4*>(dout + row * ld);
  const uint4* osrc = reinterpret_cast<const uint4*>(out + row * ld);
  uint4* edst = reinterpret_cast<uint4*>(e + row * lde);
  float acc = 0.f;
  // 8 columns (16 bytes of each tensor) per step: pairs p .. p+3 of one head, whose cos/sin
  // are 4 consecutive floats of the table row
  auto step = [&](int64_t v, const uint4 du, const uint4 ou) {
    const uint32_t dw[4] = {du.x, du.y, du.z, du.w}, ow[4] = {ou.x, ou.y, ou.z, ou.w};
    const int col = (int)(v << 3);
    float cv[4] = {1.f, 1.f, 1.f, 1.f}, sv[4] = {0.f, 0.f, 0.f, 0.f};
    if (col < rope_ncols) {
      const int64_t t = (int64_t)pos * half + ((col % head_dim) >> 1);
      const float4 c4 = __ldg(reinterpret_cast<const float4*>(cs + t));
      const float4 s4 = __ldg(reinterpret_cast<const float4*>(sn + t));
      cv[0] = c4.x; cv[1] = c4.y; cv[2] = c4.z; cv[3] = c4.w;
      sv[0] = s4.x; sv[1] = s4.y; sv[2] = s4.z; sv[3] = s4.w;
    }
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float x0 = __uint_as_float(dw[k] << 16), x1 = __uint_as_float(dw[k] & 0xFFFF0000u);
      acc = fmaf(x0, __uint_as_float(ow[k] << 16), fmaf(x1, __uint_as_float(ow[k] & 0xFFFF0000u), acc));
      const float y0 = x0 * cv[k] + x1 * sv[k], y1 = x1 * cv[k] - x0 * sv[k];
      __nv_bfloat162 b = __floats2bfloat162_rn(rr * y0, rr * y1);
      o[k] = *reinterpret_cast<uint32_t*>(&b);
    }
    edst[v] = make_uint4(o[0], o[1], o[2], o[3]);
  };
  const int64_t nv = N >> 3;
  for (int64_t v = lane; v < nv; v += 64) {   // two steps' loads in flight
    const bool two = v + 32 < nv;
    const uint4 d0 = __ldcs(dsrc + v), o0 = __ldcs(osrc + v);
    uint4 d1 = make_uint4(0, 0, 0, 0), o1 = d1;
    if (two) {
      d1 = __ldcs(dsrc + v + 32);
      o1 = __ldcs(osrc + v + 32);
    }
    step(v, d0, o0);
    if (two) step(v + 32, d1, o1);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) c[row] = rr * rr * acc * inv_h;
}

cudaError_t launch_rope_bwd(const void* dout, const void* out, int64_t M, int64_t N, int64_t ld, const float* r,
                            const float* cs, const float* sn, int seq_len, int head_dim, int rope_ncols, int64_t H,
                            void* e, int64_t lde, float* c, cudaStream_t s) {
  const int rows_per_block = 8;
  const int64_t blocks = (M + rows_per_block - 1) / rows_per_block;
  launch_k(rope_bwd_kernel, (unsigned)blocks, 32 * rows_per_block, s, 
      static_cast<const __nv_bfloat16*>(dout), static_cast<const __nv_bfloat16*>(out), M, N, ld, r, cs, sn, seq_len,
      head_dim, rope_ncols, 1.0f / (float)H, static_cast<__nv_bfloat16*>(e), lde, c);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- cross-entropy combine
// The light reduce of the per-tile online-softmax states (m_t, s_t = sum over the tile of
// exp(x - m_t)): per row, lse = log(sum_t s_t exp(m_t)); loss = lse - logit[target] (NaN for
// a target outside [0, V)).  A CTA takes 32 rows (one per lane, so each load of a warp reads
// 128 contiguous bytes) and splits the tiles among its 8 warps: warp w folds tiles w, w + 8,
// ... into a running (max, scaled sum), four tiles' loads in flight, one pass over the states;
// the 8 warps' states are then merged in warp order (deterministic).  (One thread per row
// walking all tiles twice ran at 0.45 TB/s: 64 CTAs for 16384 rows, one load in flight each.)
__device__ __forceinline__ void lse_merge(float& m, float& s, float pm, float ps) {
  if (!(pm > -INFINITY)) return;   // a state with no column
  const float mn = fmaxf(m, pm);
  s = s * __expf(m - mn) + ps * __expf(pm - mn);
  m = mn;
}
constexpr int XR_WARPS = 8;
__global__ void __launch_bounds__(32 * XR_WARPS)
    xent_reduce_kernel(const float* __restrict__ Pm, const float* __restrict__ Ps, int64_t ld, int nparts, int64_t M,
                       const float* __restrict__ T, const int* __restrict__ targets, int64_t V,
                       float* __restrict__ lse, float* __restrict__ loss) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  __shared__ float st_m[XR_WARPS][32], st_s[XR_WARPS][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t i = (int64_t)blockIdx.x * 32 + lane;
  float m = -INFINITY, s = 0.f;
  if (i < M) {
    int t = w;
    for (; t + 3 * XR_WARPS < nparts; t += 4 * XR_WARPS) {
      float pm[4], ps[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        pm[k] = __ldg(Pm + (int64_t)(t + k * XR_WARPS) * ld + i);
        ps[k] = __ldg(Ps + (int64_t)(t + k * XR_WARPS) * ld + i);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) lse_merge(m, s, pm[k], ps[k]);
    }
    for (; t < nparts; t += XR_WARPS) lse_merge(m, s, __ldg(Pm + (int64_t)t * ld + i), __ldg(Ps + (int64_t)t * ld + i));
  }
  st_m[w][lane] = m;
  st_s[w][lane] = s;
  __syncthreads();
  if (w == 0 && i < M) {
    float mm = st_m[0][lane], ss = st_s[0][lane];
#pragma unroll
    for (int g = 1; g < XR_WARPS; ++g) lse_merge(mm, ss, st_m[g][lane], st_s[g][lane]);
    const float l = mm + __logf(ss);
    lse[i] = l;
    const int tg = __ldg(targets + i);
    loss[i] = (tg >= 0 && tg < V) ? l - __ldg(T + i) : __int_as_float(0x7fc00000);
  }
}

// Mean of n floats by one block: strided partial sums in fixed order, then a fixed tree.
__global__ void mean_kernel(const float* __restrict__ x, int64_t n, float* __restrict__ out) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  __shared__ float red[1024];
  float s = 0.f;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) s += x[i];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) out[0] = red[0] / (float)n;
}

cudaError_t launch_xent_reduce(const float* Pm, const float* Ps, int64_t ld, int nparts, int64_t M, const float* T,
                               const int* targets, int64_t V, float* lse, float* loss, float* mean, cudaStream_t s) {
  launch_k(xent_reduce_kernel, (unsigned)((M + 31) / 32), 32 * XR_WARPS, s, Pm, Ps, ld, nparts, M, T, targets, V, lse,
           loss);
  if (mean) launch_k(mean_kernel, 1, 1024, s, loss, M, mean);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- column reduce
// Block = 32 columns x 32 row-groups; each thread sums a strided subset of the blocks in a
// fixed order (two loads in flight), then the 32 group sums are added in order
// (deterministic).
__global__ void col_reduce_kernel(const float* __restrict__ parts, int64_t nblocks, int64_t N, int64_t ld,
                                  float* __restrict__ out) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  __shared__ float red[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int64_t j = (int64_t)blockIdx.x * 32 + tx;
  // thread (ty, tx) sums rows ty, ty + 32, ... of column j: row ty + 32 i into running sum i % 8
  // (eight loads in flight), the rows left over into sum 0, then ((0 + 1) + (2 + 3)) + ((4 + 5) +
  // (6 + 7)); the 32 threads of a column are added in ty order
  float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (j < N) {
    int64_t b = ty;
    for (; b + 7 * 32 < nblocks; b += 8 * 32) {
#pragma unroll
      for (int k = 0; k < 8; ++k) s[k] += __ldg(parts + (b + 32 * k) * ld + j);
    }
    for (; b < nblocks; b += 32) s[0] += __ldg(parts + b * ld + j);
  }
  red[ty][tx] = ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
  __syncthreads();
  if (ty == 0 && j < N) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) t += red[k][tx];
    out[j] = t;
  }
}

cudaError_t launch_col_reduce(const float* parts, int64_t nblocks, int64_t N, int64_t ld, float* out,
                              cudaStream_t s) {
  const int64_t blocks = (N + 31) / 32;
  launch_k(col_reduce_kernel, (unsigned)blocks, 1024, s, parts, nblocks, N, ld, out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- gain fold
// W'[n, k] = bf16(W[n, k] * g[k]); 8 elements (16 bytes) per thread per step, grid-stride.
__global__ void fold_gain_kernel(const __nv_bfloat16* __restrict__ W, int64_t N, int64_t K, int64_t ld_in,
                                 const float* __restrict__ g, float inv_scale, __nv_bfloat16* __restrict__ Wo,
                                 int64_t ld_out) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int64_t kv = K >> 3;
  const int64_t total = N * kv;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total; v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = v / kv, k = (v - n * kv) << 3;
    const uint4 u = __ldcs(reinterpret_cast<const uint4*>(W + n * ld_in + k));
    const float4 g0 = __ldg(reinterpret_cast<const float4*>(g + k));
    const float4 g1 = __ldg(reinterpret_cast<const float4*>(g + k + 4));
    const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __uint_as_float(w[e] << 16) * gv[2 * e] * inv_scale;
      const float hi = __uint_as_float(w[e] & 0xFFFF0000u) * gv[2 * e + 1] * inv_scale;
      __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
      o[e] = *reinterpret_cast<uint32_t*>(&b);
    }
    __stcs(reinterpret_cast<uint4*>(Wo + n * ld_out + k), make_uint4(o[0], o[1], o[2], o[3]));
  }
}

// fp32 weights: 4 elements (16 bytes) per thread per step.
__global__ void fold_gain_f32_kernel(const float* __restrict__ W, int64_t N, int64_t K, int64_t ld_in,
                                     const float* __restrict__ g, float inv_scale, float* __restrict__ Wo,
                                     int64_t ld_out) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int64_t kv = K >> 2;
  const int64_t total = N * kv;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total; v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = v / kv, k = (v - n * kv) << 2;
    const float4 w = __ldcs(reinterpret_cast<const float4*>(W + n * ld_in + k));
    const float4 gv = __ldg(reinterpret_cast<const float4*>(g + k));
    __stcs(reinterpret_cast<float4*>(Wo + n * ld_out + k),
           make_float4(w.x * gv.x * inv_scale, w.y * gv.y * inv_scale, w.z * gv.z * inv_scale,
                       w.w * gv.w * inv_scale));
  }
}

// bf16 weights to e4m3 codes of W g / out_scale: 16 elements (32 bytes in, 16 bytes out) per
// thread per step.
__global__ void fold_gain_e4m3_kernel(const __nv_bfloat16* __restrict__ W, int64_t N, int64_t K, int64_t ld_in,
                                      const float* __restrict__ g, float inv_scale, uint8_t* __restrict__ Wo,
                                      int64_t ld_out) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int64_t kv = K >> 4;
  const int64_t total = N * kv;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total; v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = v / kv, k = (v - n * kv) << 4;
    const uint4 u0 = __ldcs(reinterpret_cast<const uint4*>(W + n * ld_in + k));
    const uint4 u1 = __ldcs(reinterpret_cast<const uint4*>(W + n * ld_in + k + 8));
    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float4 gv = __ldg(reinterpret_cast<const float4*>(g + k + 4 * e));
      const float a0 = __uint_as_float(w[2 * e] << 16) * gv.x * inv_scale;
      const float a1 = __uint_as_float(w[2 * e] & 0xFFFF0000u) * gv.y * inv_scale;
      const float a2 = __uint_as_float(w[2 * e + 1] << 16) * gv.z * inv_scale;
      const float a3 = __uint_as_float(w[2 * e + 1] & 0xFFFF0000u) * gv.w * inv_scale;
      o[e] = (uint32_t)ptx::cvt_e4m3x2(a0, a1) | ((uint32_t)ptx::cvt_e4m3x2(a2, a3) << 16);
    }
    __stcs(reinterpret_cast<uint4*>(Wo + n * ld_out + k), make_uint4(o[0], o[1], o[2], o[3]));
  }
}

cudaError_t launch_fold_gain(const void* W, int64_t N, int64_t K, int64_t ld_in, const float* g, float inv_scale,
                             void* W_out, int64_t ld_out, int out_kind, cudaStream_t s, int sms) {
  const int threads = 256;
  const int shift = out_kind == FOLD_OUT_F32 ? 2 : out_kind == FOLD_OUT_E4M3 ? 4 : 3;
  const int64_t need = (N * (K >> shift) + threads - 1) / threads;
  const int64_t cap = (int64_t)sms * 8;
  const int64_t blocks = need < cap ? need : cap;
  if (blocks <= 0) return cudaSuccess;
  if (out_kind == FOLD_OUT_F32)
    launch_k(fold_gain_f32_kernel, (unsigned)blocks, threads, s, static_cast<const float*>(W), N, K, ld_in, g,
             inv_scale, static_cast<float*>(W_out), ld_out);
  else if (out_kind == FOLD_OUT_E4M3)
    launch_k(fold_gain_e4m3_kernel, (unsigned)blocks, threads, s, static_cast<const __nv_bfloat16*>(W), N, K, ld_in,
             g, inv_scale, static_cast<uint8_t*>(W_out), ld_out);
  else
    launch_k(fold_gain_kernel, (unsigned)blocks, threads, s, static_cast<const __nv_bfloat16*>(W), N, K, ld_in, g,
             inv_scale, static_cast<__nv_bfloat16*>(W_out), ld_out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- RoPE table
__global__ void rope_table_kernel(int seq_len, int half, double base, int head_dim, float* __restrict__ c,
                                  float* __restrict__ s) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)seq_len * half) return;
  const int pos = (int)(idx / half), p = (int)(idx % half);
  const double inv_freq = pow(base, -2.0 * (double)p / (double)head_dim);
  double sn, cs;
  sincos((double)pos * inv_freq, &sn, &cs);
  c[idx] = (float)cs;
  s[idx] = (float)sn;
}

// ---------------------------------------------------------------- e4m3 quantisation
// Q[i, j] = e4m3(X[i, j] * inv_scale) (nearest even, saturating); 16 elements (32 bytes in,
// 16 bytes out) per thread per step, grid-stride; optional running max of |X|.
__global__ void quantize_e4m3_kernel(const __nv_bfloat16* __restrict__ X, int64_t M, int64_t N, int64_t ldx,
                                     float inv_scale, uint8_t* __restrict__ Q, int64_t ldq,
                                     unsigned int* __restrict__ amax) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int64_t nv = N >> 4;
  const int64_t total = M * nv;
  float m = 0.f;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total; v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = v / nv, j = (v - i * nv) << 4;
    const uint4* src = reinterpret_cast<const uint4*>(X + i * ldx + j);
    const uint4 u0 = __ldcs(src), u1 = __ldcs(src + 1);
    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a0 = __uint_as_float(w[2 * e] << 16), a1 = __uint_as_float(w[2 * e] & 0xFFFF0000u);
      const float a2 = __uint_as_float(w[2 * e + 1] << 16), a3 = __uint_as_float(w[2 * e + 1] & 0xFFFF0000u);
      m = fmaxf(m, fmaxf(fmaxf(fabsf(a0), fabsf(a1)), fmaxf(fabsf(a2), fabsf(a3))));
      o[e] = (uint32_t)ptx::cvt_e4m3x2(a0 * inv_scale, a1 * inv_scale) |
             ((uint32_t)ptx::cvt_e4m3x2(a2 * inv_scale, a3 * inv_scale) << 16);
    }
    __stcs(reinterpret_cast<uint4*>(Q + i * ldq + j), make_uint4(o[0], o[1], o[2], o[3]));
  }
  if (amax) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0 && m > 0.f) atomicMax(amax, __float_as_uint(m));   // |x| orders as its bits
  }
}

cudaError_t launch_quantize_e4m3(const void* X, int64_t M, int64_t N, int64_t ldx, float inv_scale, void* Q,
                                 int64_t ldq, float* amax, cudaStream_t s, int sms) {
  const int threads = 256;
  const int64_t total = M * (N >> 4);
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  if (blocks < 1) blocks = 1;
  launch_k(quantize_e4m3_kernel, (unsigned)blocks, threads, s, reinterpret_cast<const __nv_bfloat16*>(X), M, N, ldx,
                                                            inv_scale, reinterpret_cast<uint8_t*>(Q), ldq,
                                                            reinterpret_cast<unsigned int*>(amax));
  return cudaGetLastError();
}

// NVFP4 quantiser: one thread per block of 16 elements of a row (32 bytes read, 8 bytes of
// codes and one scale byte written); rows from R up to the next multiple of 128 get zero
// scales.
__global__ void quantize_nvfp4_kernel(const __nv_bfloat16* __restrict__ X, int64_t R, int64_t K, int64_t ldx, float s,
                                      uint8_t* __restrict__ Q, int64_t ldq, uint8_t* __restrict__ sf,
                                      unsigned int* __restrict__ amax) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int64_t nb = K >> 4, kc = K >> 6;
  const int64_t rpad = (R + 127) / 128 * 128;
  const int64_t total = rpad * nb;
  float m = 0.f;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total; v += (int64_t)gridDim.x * blockDim.x) {
    const int64_t i = v / nb, b = v - i * nb;
    uint32_t code = 0;
    if (i < R) {
      const uint4* src = reinterpret_cast<const uint4*>(X + i * ldx + 16 * b);
      const uint4 u0 = __ldcs(src), u1 = __ldcs(src + 1);
      const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
      float x[16];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        x[2 * e] = __uint_as_float(w[e] << 16);
        x[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
        m = fmaxf(m, fmaxf(fabsf(x[2 * e]), fabsf(x[2 * e + 1])));
      }
      uint32_t q[2];
      code = nvfp4_block16(x, s, q);
      __stcs(reinterpret_cast<uint2*>(Q + i * ldq + 8 * b), make_uint2(q[0], q[1]));
    }
    sf[sf_offset(i, b, kc)] = (uint8_t)code;
  }
  if (amax) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0 && m > 0.f) atomicMax(amax, __float_as_uint(m));
  }
}

cudaError_t launch_quantize_nvfp4(const void* X, int64_t R, int64_t K, int64_t ldx, float s, void* Q, int64_t ldq_bytes,
                                  uint8_t* sf, float* amax, cudaStream_t st, int sms) {
  const int threads = 256;
  const int64_t total = (R + 127) / 128 * 128 * (K >> 4);
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  if (blocks < 1) blocks = 1;
  launch_k(quantize_nvfp4_kernel, (unsigned)blocks, threads, st, reinterpret_cast<const __nv_bfloat16*>(X), R, K, ldx,
           s, reinterpret_cast<uint8_t*>(Q), ldq_bytes, sf, reinterpret_cast<unsigned int*>(amax));
  return cudaGetLastError();
}

// Transposed NVFP4 quantiser: X [R, C] bf16 is quantised along its columns, into Q = X^T
// ([C, R] codes, blocks of 16 consecutive rows of X), the operand layout of a GEMM that
// contracts over R (a weight gradient contracts over the tokens).  With SWIGLU, X is the saved
// [G | U] ([R, 2C]) and the quantised value is silu(G) U.  With ROWS, the same pass also writes
// X quantised along its rows (Qr [R, C], blocks of 16 consecutive columns), so that a tensor
// needed both ways is read once.
// Persistent CTAs walk tiles of 128 rows x 128 columns: the block scales of a tile are then
// whole 512-byte atoms in both directions (128 rows of the destination by four blocks of 16
// along its K).  Every output of a tile is staged in shared memory and leaves in 16-byte
// stores: each destination row's codes as 64 contiguous bytes, the scales as two contiguous
// atoms.  (Single-byte scale stores straight from the quantising threads cost more than the
// whole read.)
//   - A tile's 16-byte loads (8 consecutive values of a row per thread, 8 per thread) are
//     issued into registers while the previous tile is quantised.
//   - Along the rows the values never leave the registers: the two threads holding a block of
//     16 exchange their maxima with one shuffle, and each stages its 8 codes (4 bytes).
//   - Along the columns the tile is staged in shared memory (as bf16, or fp32 for silu(G) U);
//     a warp reads 64 consecutive columns of a row, two per thread in one 4- or 8-byte load,
//     conflict-free, and a thread quantises two 16-row blocks of each of its two columns.
constexpr int QT_ROWS = 128, QT_COLS = 128;

// The transposed pass's own NVFP4 decisions, cheaper than nvfp4_block16's (the pass is bound
// by instruction issue, not by DRAM, so every instruction per element counts):
//   sf = e4m3(amax * inv6s), inv6s = 1 / (6 s) rounded once on the host, and
//   q = e2m1(x * rcp(sf s)) with the hardware's approximate reciprocal (at most one ulp from
// 1 / (sf s)).  Both stay within a few fp32 roundings of the exact quotients, so a decision
// can differ from exact arithmetic only for a value that close to a rounding midpoint.
__device__ __forceinline__ float qt_rcp(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
// e4m3 block scale of a block with maximum magnitude amax (its byte in *code), and the
// multiplier that takes the block's values to e2m1 code units (0 for a zero scale)
__device__ __forceinline__ float qt_scale(float amax, float inv6s, float s, uint32_t* code) {
  const uint16_t code2 = ptx::cvt_e4m3x2(amax * inv6s, 0.0f);
  float sfv, zero;
  ptx::e4m3x2_to_f32(code2, sfv, zero);
  *code = code2 & 0xFFu;
  const float d = sfv * s;
  return d > 0.f ? qt_rcp(d) : 0.f;
}
// codes of 8 values times the multiplier rd (element j in nibble j)
__device__ __forceinline__ uint32_t qt_codes8(const float* x, float rd) {
  float y[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) y[j] = x[j] * rd;
  return ptx::cvt_e2m1x8(y);
}

template <bool SWIGLU, bool ROWS>
__global__ void __launch_bounds__(256, SWIGLU ? 2 : 3) quantize_nvfp4_t_kernel(const __nv_bfloat16* __restrict__ X, int64_t R,
                                                                  int64_t C, int64_t ldx, float s, float inv6s,
                                                                  uint8_t* __restrict__ Q, int64_t ldq,
                                                                  uint8_t* __restrict__ sf, uint8_t* __restrict__ Qr,
                                                                  int64_t ldqr, uint8_t* __restrict__ sfr,
                                                                  unsigned int* __restrict__ amax) {
  using T = typename std::conditional<SWIGLU, float, __nv_bfloat16>::type;
  extern __shared__ __align__(16) uint8_t qt_smem[];
  T* tile = reinterpret_cast<T*>(qt_smem);                              // [QT_ROWS][QT_COLS]
  uint8_t* colq = qt_smem + sizeof(T) * QT_ROWS * QT_COLS;               // [QT_COLS][64 B]: Q's rows
  uint8_t* colsf = colq + QT_COLS * QT_ROWS / 2;                         // two atoms of Q's scales
  uint8_t* rowq = colsf + 1024;                                          // [QT_ROWS][64 B]: Qr's rows
  uint8_t* rowsf = rowq + QT_ROWS * QT_COLS / 2;                         // two atoms of Qr's scales
  constexpr int NP = QT_ROWS * QT_COLS / 8 / 256;   // 16-byte units of X per thread and tile
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int64_t col_tiles = C / QT_COLS;   // C is a multiple of 128
  const int64_t tiles = ((R + QT_ROWS - 1) / QT_ROWS) * col_tiles;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, u = t % 16;
  float m = 0.f;
  uint4 a[NP], b[SWIGLU ? NP : 1];
  auto issue = [&](int64_t tl) {
    const int64_t r0 = (tl / col_tiles) * QT_ROWS, c0 = (tl % col_tiles) * QT_COLS;
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      const int64_t gr = r0 + t / 16 + 16 * p, gc = c0 + 8 * u;
      const bool in = gr < R;   // rows past R (R is a multiple of 64) read as zeros
      a[p] = in ? __ldcs(reinterpret_cast<const uint4*>(X + gr * ldx + gc)) : make_uint4(0, 0, 0, 0);
      if constexpr (SWIGLU)
        b[p] = in ? __ldcs(reinterpret_cast<const uint4*>(X + gr * ldx + C + gc)) : make_uint4(0, 0, 0, 0);
    }
  };
  int64_t tl = blockIdx.x;
  if (tl < tiles) issue(tl);
  for (; tl < tiles; tl += gridDim.x) {
    const int64_t r0 = (tl / col_tiles) * QT_ROWS, c0 = (tl % col_tiles) * QT_COLS;
    __syncthreads();   // the previous tile's shared tile and staged outputs are no longer read
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      const int row = t / 16 + 16 * p;
      const uint32_t w[4] = {a[p].x, a[p].y, a[p].z, a[p].w};
      float v[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        v[2 * k] = __uint_as_float(w[k] << 16);
        v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
      }
      if constexpr (SWIGLU) {
        const uint32_t wu[4] = {b[p].x, b[p].y, b[p].z, b[p].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          v[2 * k] = silu_f(v[2 * k]) * __uint_as_float(wu[k] << 16);
          v[2 * k + 1] = silu_f(v[2 * k + 1]) * __uint_as_float(wu[k] & 0xFFFF0000u);
        }
        float4* dst = reinterpret_cast<float4*>(tile + row * QT_COLS + 8 * u);
        dst[0] = make_float4(v[0], v[1], v[2], v[3]);
        dst[1] = make_float4(v[4], v[5], v[6], v[7]);
      } else {
        *reinterpret_cast<uint4*>(tile + row * QT_COLS + 8 * u) = a[p];
      }
      float m8 = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) m8 = fmaxf(m8, fabsf(v[k]));
      m = fmaxf(m, m8);
      if constexpr (ROWS) {   // along the rows, from the registers: threads t, t ^ 1 hold a block
        const float m16 = fmaxf(m8, __shfl_xor_sync(0xffffffffu, m8, 1));
        uint32_t code;
        const float rd = qt_scale(m16, inv6s, s, &code);
        *reinterpret_cast<uint32_t*>(rowq + row * 64 + 4 * u) = qt_codes8(v, rd);
        if ((u & 1) == 0) {
          const int kb = u >> 1;   // block of 16 along the row, 0..7
          rowsf[(kb >> 2) * 512 + 16 * (row % 32) + 4 * (row / 32) + (kb & 3)] = (uint8_t)code;
        }
      }
    }
    __syncthreads();
    const int64_t nx = tl + gridDim.x;   // the next tile's loads fly while this one is quantised
    if (nx < tiles) issue(nx);
    {   // along the columns: warp w takes the column pairs (2 cp, 2 cp + 1), cp = 32 (w % 2) +
        // lane (a warp's loads cover 128 or 256 contiguous bytes of a row, conflict-free), and
        // the two 16-row blocks 2 j, 2 j + 1, j = w / 2: 32 rows of each of its two columns
      const int cp = 32 * (warp & 1) + lane, j = warp >> 1;
      uint32_t q[2][4], code[2][2];   // [column h][...]: codes of blocks 2 j, 2 j + 1; their scales
#pragma unroll
      for (int i = 0; i < 2; ++i) {   // block 2 j + i: 16 rows of both columns
        if constexpr (SWIGLU) {
          float x[2][16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 v2 = *reinterpret_cast<const float2*>(tile + (32 * j + 16 * i + k) * QT_COLS + 2 * cp);
            x[0][k] = v2.x;
            x[1][k] = v2.y;
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float am = 0.f;
#pragma unroll
            for (int k = 0; k < 16; ++k) am = fmaxf(am, fabsf(x[h][k]));
            const float rd = qt_scale(am, inv6s, s, &code[h][i]);
            q[h][2 * i] = qt_codes8(x[h], rd);
            q[h][2 * i + 1] = qt_codes8(x[h] + 8, rd);
          }
        } else {   // the two columns' bf16 values stay packed until each is quantised
          uint32_t w2[16];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            w2[k] = *reinterpret_cast<const uint32_t*>(tile + (32 * j + 16 * i + k) * QT_COLS + 2 * cp);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float x[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) x[k] = __uint_as_float(h ? (w2[k] & 0xFFFF0000u) : (w2[k] << 16));
            float am = 0.f;
#pragma unroll
            for (int k = 0; k < 16; ++k) am = fmaxf(am, fabsf(x[k]));
            const float rd = qt_scale(am, inv6s, s, &code[h][i]);
            q[h][2 * i] = qt_codes8(x, rd);
            q[h][2 * i + 1] = qt_codes8(x + 8, rd);
          }
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {   // column c = 2 cp + h
        const int c = 2 * cp + h;
        // blocks 2 j, 2 j + 1 of column c form 16-byte unit j of row c, its place XOR-swizzled
        // by bits 1-2 of c (blocks past R are staged, never stored)
        *reinterpret_cast<uint4*>(colq + c * 64 + 16 * (j ^ ((c >> 1) & 3))) =
            make_uint4(q[h][0], q[h][1], q[h][2], q[h][3]);
        // their scales: bytes 2 (j % 2) and 2 (j % 2) + 1 of row c's group in atom j / 2
        *reinterpret_cast<uint16_t*>(colsf + (j >> 1) * 512 + 16 * (c % 32) + 4 * (c / 32) + 2 * (j & 1)) =
            (uint16_t)(code[h][0] | (code[h][1] << 8));
      }
    }
    __syncthreads();
    // the staged outputs, in 16-byte stores: 4 units per destination row, 32 per atom
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = t + 256 * k, c = i >> 2, j = i & 3;
      if (r0 + 32 * j < R)
        __stcs(reinterpret_cast<uint4*>(Q + (c0 + c) * ldq + r0 / 2 + 16 * j),
               *reinterpret_cast<const uint4*>(colq + c * 64 + 16 * (j ^ ((c >> 1) & 3))));
      if constexpr (ROWS)   // R is a multiple of 128 here
        __stcs(reinterpret_cast<uint4*>(Qr + (r0 + c) * ldqr + c0 / 2 + 16 * j),
               *reinterpret_cast<const uint4*>(rowq + c * 64 + 16 * j));
    }
    if (t < 64) {
      const int at = t >> 5, off = 16 * (t & 31);
      if (r0 + 64 * at < R)
        __stcs(reinterpret_cast<uint4*>(sf + ((c0 / 128) * (R / 64) + r0 / 64 + at) * 512 + off),
               *reinterpret_cast<const uint4*>(colsf + at * 512 + off));
    } else if (ROWS && t < 128) {
      const int at = (t - 64) >> 5, off = 16 * (t & 31);
      __stcs(reinterpret_cast<uint4*>(sfr + ((r0 / 128) * (C / 64) + c0 / 64 + at) * 512 + off),
             *reinterpret_cast<const uint4*>(rowsf + at * 512 + off));
    }
  }
  if (amax) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0 && m > 0.f) atomicMax(amax, __float_as_uint(m));
  }
}

cudaError_t launch_quantize_nvfp4_t(const void* X, int64_t R, int64_t C, int64_t ldx, bool swiglu, float s, void* Q,
                                    int64_t ldq_bytes, uint8_t* sf, void* Qr, int64_t ldqr_bytes, uint8_t* sfr,
                                    float* amax, cudaStream_t st, int sms) {
  const int64_t tiles = ((R + QT_ROWS - 1) / QT_ROWS) * ((C + QT_COLS - 1) / QT_COLS);
  if (tiles <= 0) return cudaSuccess;
  // the tile, then the staged outputs: Q's codes and scales, Qr's codes and scales
  const size_t smem = (swiglu ? sizeof(float) : sizeof(__nv_bfloat16)) * QT_ROWS * QT_COLS +
                      (QT_ROWS * QT_COLS / 2 + 1024) * (Qr ? 2 : 1);
  auto go = [&](auto kernel) {
    if (smem > 48 * 1024) {   // the fp32 tile of silu(G) U: above the default dynamic limit
      const cudaError_t ae = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (ae != cudaSuccess) return ae;
    }
    // persistent: as many CTAs as fit on every SM at once
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, smem) != cudaSuccess || per_sm < 1) {
      cudaGetLastError();
      per_sm = 1;
    }
    const int64_t grid = tiles < (int64_t)sms * per_sm ? tiles : (int64_t)sms * per_sm;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = g_launch_overlap ? 1 : 0;
    const float inv6s = (float)(1.0 / (6.0 * (double)s));
    return cudaLaunchKernelEx(&cfg, kernel, reinterpret_cast<const __nv_bfloat16*>(X), R, C, ldx, s, inv6s,
                              reinterpret_cast<uint8_t*>(Q), ldq_bytes, sf, reinterpret_cast<uint8_t*>(Qr), ldqr_bytes,
                              sfr, reinterpret_cast<unsigned int*>(amax));
  };
  cudaError_t e;
  if (swiglu)
    e = Qr ? go(quantize_nvfp4_t_kernel<true, true>) : go(quantize_nvfp4_t_kernel<true, false>);
  else
    e = Qr ? go(quantize_nvfp4_t_kernel<false, true>) : go(quantize_nvfp4_t_kernel<false, false>);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_rope_table(int seq_len, int head_dim, double base, float* cos_out, float* sin_out,
                              cudaStream_t s) {
  const int half = head_dim / 2;
  const int64_t n = (int64_t)seq_len * half;
  const int threads = 256;
  launch_k(rope_table_kernel, (unsigned)((n + threads - 1) / threads), threads, s, seq_len, half, base, head_dim,
                                                                                 cos_out, sin_out);
  return cudaGetLastError();
}

}  // namespace coda
