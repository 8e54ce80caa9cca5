// Persistent tcgen05 GEMM with a programmable epilogue (sm_103a).
//
// What it computes (one launch):  out = epilogue(acc),  acc[M, N] = A[M, K] . B[N, K]^T
// with fp32 accumulation in TMEM.  This is the "fixed GEMM mainloop + composable
// epilogue" split the CODA pages describe: the mainloop is written once; the epilogue
// runs while the output tile is still on chip, before its single store to HBM
// ("CODA: new research optimizes Transformer training with GEMM-epilogue programming",
// kucoin.com news flash, sections "El epílogo esconde un tesoro" and "Cinco bloques y un
// lenguaje LEGO").  The pages picture the tile in registers; on this GPU it lives in
// tensor memory (TMEM) and is read back in 32-column chunks by the epilogue warps.
//
// Structure (CTA pairs: clusters of two CTAs on two SMs, persistent over 256 x 256 output
// tiles; each CTA owns 128 rows of the tile):
//   warp 0      TMA producer: this CTA's 128 rows of A and 128 rows of B per k-block into a
//               STAGES-deep shared-memory ring (both CTAs' copies complete on the leader's
//               barrier)
//   warp 1      TMEM allocation; in the leader CTA, single-thread tcgen05.mma.cta_group::2
//               issue (256 x 256 x 32 bytes of K per instruction) into one of two TMEM
//               accumulators (2 x 256 columns in each CTA)
//   warps 2..5  epilogue: tcgen05.ld (thread = output row), the epilogue program, row /
//               column partial reductions, cast, swizzled staging in shared memory and
//               TMA stores; side inputs (residual, saved activations) arrive by TMA.
//   warps 6..9  NVFP4 only: block scales from shared memory into TMEM with tcgen05.st, one
//               warp per TMEM lane quarter (NVFP4 tiles keep one accumulator; the other
//               TMEM columns hold the scales of the ring's stages).
// The two TMEM accumulators let tile t+1's mainloop run under tile t's epilogue.  The
// launch carries a programmatic dependency on the previous kernel of the stream (see
// griddep_wait in coda_ptx.cuh).
//
// Every wait is bounded (global timer).  On expiry the waiting thread records a site
// code in a device status word, raises a CTA-wide abort flag, every role leaves its loop,
// copies in flight are drained with a short bounded wait, TMEM is freed and the kernel
// returns; the host reads the status word.  Nothing traps.
#pragma once
#include <atomic>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "coda_ptx.cuh"

namespace coda {

// ----------------------------------------------------------------------- constants
constexpr int BM = 128;                               // tile rows = TMEM lanes
constexpr int UMMA_N = 256;                           // MMA N = B tile rows
constexpr int BK_BYTES = 128;                         // K bytes per 128B swizzle row (a stage holds one or two)
constexpr int KSTEPS = 4;                             // MMAs per stage, 32 bytes of K each
constexpr int A_STAGE_BYTES = BM * BK_BYTES;          // 16 KB: this CTA's 128 rows of A
constexpr int TMEM_COLS = 2 * UMMA_N;                 // two fp32 accumulators
constexpr int NUM_EPI_WARPS = 4;
constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr int MAX_SMEM = 232448;                      // 227 KB opt-in per CTA

enum : int { DT_F32 = 0, DT_BF16 = 1, DT_E4M3 = 2, DT_E2M1 = 3 };
__host__ __device__ constexpr int dt_bytes(int dt) { return dt == DT_F32 ? 4 : dt == DT_BF16 ? 2 : 1; }
// bytes of one 32 x 32 staging block (e2m1: two codes per byte)
__host__ __device__ constexpr int slot_bytes(int dt) { return dt == DT_E2M1 ? 512 : 32 * 32 * dt_bytes(dt); }

// KIND_NVFP4: e2m1 operands packed two per byte along K, one ue4m3 scale per 16 K elements
// (block-scaled MMA, scales stored into TMEM by scale warps), fp32 tensor scales in the epilogue.
enum : int { KIND_BF16 = 0, KIND_TF32 = 1, KIND_E4M3 = 2, KIND_NVFP4 = 3 };

// NVFP4 block scales in memory: atoms of 128 rows x 4 blocks of 16 K elements (512 bytes).
// Atom (row / 128, kb / 4) sits at ((row / 128) * kc + kb / 4) * 512, kc = K / 64 atoms per
// 128-row block; inside an atom, row r is at byte 16 (r % 32) + 4 ((r % 128) / 32) and block
// kb at + kb % 4: the 16 bytes at 16 i hold rows i + 32 q (q = 0..3), the order of the
// 4-column groups from which the block-scaled MMA reads row r's scales (lane r, column
// (r % 128) / 32).
__host__ __device__ constexpr long long sf_offset(long long row, long long kb, long long kc) {
  return ((row / 128) * kc + kb / 4) * 512 + 16 * (row % 32) + 4 * ((row % 128) / 32) + kb % 4;
}

// Compiled epilogue programs (the host maps an op list onto one of these).
enum : int {
  EPI_STORE = 0,       // out = ts * acc [* g_col]
  EPI_RESID = 1,       // out = ts * acc + R            [+ row partial sum of squares of out]
                       //   [+ aux = out * g_col: the RMSNorm gain broadcast along the tile]
  EPI_ROWSCALE = 2,    // out = ts * r_row * acc
  EPI_SWIGLU = 3,      // Z = ts * r_row * acc (gate | up halves); out = silu(Zg) * Zu * os
                       //   [+ saved Z, + amax |silu(Zg) * Zu|]
  EPI_ROPE = 4,        // out = rope(ts * r_row * acc) on the first rope_ncols columns
  EPI_SWIGLU_BWD = 5,  // dA = ts * acc; e = r_row * [dA * Zu * silu'(Zg) | dA * silu(Zg)]; row partial
                       //   sum e . Z; e4m3 out: codes of e * os, partial of the dequantised e, amax |e|
  EPI_RMSBWD = 6,      // t = ts * acc; out = g_col * t - c_row * h [+ dY] (g = 1 without F_COLSCALE);
                       //   column partial sum h * t (F_COLPART)
  EPI_XENT = 7,        // z = ts * r_row * acc (logits, never stored): per tile and row the online
                       //   state (max_j z, sum_j exp(z - max)) and the target's logit
  EPI_XENT_BWD = 8,    // z as above; e = r_row * os * (exp(z - lse_row) - [j == target_row]);
                       //   row partial sum e . z
};

enum : int {
  F_PARTIAL = 1,    // write row partials (EPI_RESID)
  F_AMAX = 4,       // accumulate amax (EPI_SWIGLU)
  F_COLSCALE = 8,   // multiply by col_scale (EPI_STORE)
  F_ROWSCALE = 16,  // multiply by row_scale (EPI_SWIGLU / EPI_ROPE / EPI_ROWSCALE / EPI_SWIGLU_BWD)
  F_NO_SIDE1 = 32,  // EPI_RMSBWD without the dY side input
  F_COLPART = 64,   // write column partials (EPI_RMSBWD)
  F_AB_READY = 128, // A and B are not written by the previous kernel of the stream
  F_A_STREAM = 256, // A's loads carry an evict_first policy (see the host's tile order)
  F_INJECT_SKIP = 1 << 30,  // test hook: the producer drops its first k-block
  F_INJECT_RANK0 = 1 << 29, // test hook: only the pair's leader drops it
  F_INJECT_RANK1 = 1 << 28, // test hook: only the pair's second CTA drops it
};

// Device status word: 0 = fine; otherwise the site of the first wait that timed out.
enum : int {
  SITE_PRODUCER_EMPTY = 1,
  SITE_MMA_TMEM_EMPTY = 2,
  SITE_MMA_FULL = 3,
  SITE_EPI_TMEM_FULL = 4,
  SITE_EPI_SIDE = 5,
  SITE_SCALES_FULL = 6,   // NVFP4 scale warp / block scales in shared memory
  SITE_MMA_SCALES = 7,    // MMA / block scales in TMEM (both CTAs)
};

struct GemmParams {
  int M, N, K;          // out [M, N]; EPI_SWIGLU: N = F and B holds 2F rows (gate, then up)
  int m_tiles, n_tiles;
  int group_n;          // tile order: groups of group_n N-tiles, M-major inside a group
  int k_splits;         // split-K: each tile's K range in k_splits slices, reduce-added into out
  int kb_per_split;     // k-blocks per slice (the last slice may be shorter)
  int flags;
  int up_offset;        // EPI_SWIGLU: first up row of B / first U column of saved Z;
                        // EPI_SWIGLU_BWD: first U column of Z and of e
  float tensor_scale;   // ts above (fp8 dequantisation), 1 otherwise
  float out_scale;      // os above (1 / s_a before an e4m3 cast), 1 otherwise
  const float* row_scale;
  const float* row_coef;
  const float* col_scale;
  const float* rope_cos;  // [rope_seq_len, rope_head_dim / 2]
  const float* rope_sin;
  int rope_seq_len, rope_head_dim, rope_ncols;
  float* row_part;        // [n_tiles, row_part_ld]
  long long row_part_ld;
  float* row_part2;       // EPI_XENT: sum-exp partials, same layout as row_part (the maxima)
  float* row_out;         // EPI_XENT: [M] logit of each row's target
  const int* row_index;   // EPI_XENT / EPI_XENT_BWD: [M] target class of each row
  float* col_part;        // [4 * m_tiles, col_part_ld]
  long long col_part_ld;
  unsigned int* amax;     // fp32 bits, atomic max (non-negative values order as integers)
  float fp4_scale;        // NVFP4 output: tensor scale s of the codes
  uint8_t* out_sf;        // NVFP4 output: block scales (atom layout, kc = out_sf_kc)
  long long out_sf_kc;
  int* status;
  unsigned long long timeout_ns;
};

// Pipeline stages that fit in `free_bytes` of shared memory, at most `max_stages`.
__host__ __device__ constexpr int fit_stages(int free_bytes, int stage_bytes, int max_stages) {
  return free_bytes / stage_bytes > max_stages ? max_stages : free_bytes / stage_bytes;
}

// CG = CTAs per MMA: 1, or 2 for a CTA pair (cluster of two) issuing cta_group::2 MMAs of
// 256 x 256: each CTA holds 128 rows of A and 128 rows (N) of B per stage and receives its
// 128 accumulator rows in its own TMEM.
// UN = MMA N (B rows of a tile).  256 fills TMEM with two accumulators.  NVFP4 tiles keep
// UN = 256 with one accumulator, so that the block scales of the pipeline stages fit in TMEM
// beside it (the epilogue of a tile then runs between that tile's MMAs and the next's).
template <int KIND_, int EPI_, bool A_MN_, bool B_MN_, int OUT_DT_, int SIDE_DT_, bool AUX_, int CG_ = 2,
          int UN_ = UMMA_N>
struct GemmCfg {
  static constexpr int KIND = KIND_, EPI = EPI_, OUT_DT = OUT_DT_, SIDE_DT = SIDE_DT_, CG = CG_, UN = UN_;
  static constexpr bool A_MN = A_MN_, B_MN = B_MN_, AUX = AUX_;
  static constexpr bool FP4 = KIND == KIND_NVFP4;
  static constexpr int B_ROWS = UN / CG;                       // B rows (N) held by this CTA
  static constexpr int B_BOX = B_ROWS < 128 ? B_ROWS : 128;    // rows per B copy
  static constexpr int B_ROW_BYTES = B_ROWS * BK_BYTES;        // this CTA's B for one 128-byte row of K
  // NVFP4 block scales of a stage: one atom per MMA for this CTA's 128 rows of A, and one per
  // MMA and 128 rows of the tile's N for B (each CTA of a pair holds all of them)
  static constexpr int SF_A_BYTES = FP4 ? KSTEPS * 512 : 0;
  static constexpr int SF_B_BYTES = FP4 ? KSTEPS * 512 * (UN / 128) : 0;
  static constexpr int SB1 = A_STAGE_BYTES + B_ROW_BYTES + SF_A_BYTES + SF_B_BYTES;   // a stage of one K row
  static constexpr int PAIR_ROWS = BM * CG;                    // output rows per tile
  static constexpr int OP_BYTES = KIND == KIND_TF32 ? 4 : KIND == KIND_BF16 ? 2 : 1;
  static constexpr bool DUAL = EPI == EPI_SWIGLU;
  static constexpr int BN_OUT = DUAL ? UN / 2 : UN;  // output columns per tile
  static constexpr int NCHUNK = BN_OUT / 32;
  static constexpr int NS = EPI == EPI_RESID ? 1 : (EPI == EPI_SWIGLU_BWD || EPI == EPI_RMSBWD) ? 2 : 0;
  static constexpr int NO = EPI == EPI_SWIGLU_BWD ? 2 : EPI == EPI_XENT ? 0 : 1;   // XENT stores no tile
  static constexpr int OSLOT = slot_bytes(OUT_DT);  // one 32 x 32 staging block
  static constexpr int SSLOT = slot_bytes(SIDE_DT);
  static constexpr int XSLOT = 32 * 32 * 2;                 // aux output block (bf16)
  static constexpr int NX = AUX ? (EPI == EPI_SWIGLU ? 2 : 1) : 0;   // SwiGLU: G and U; residual: h * g
  static constexpr int OUTSET = NO * OSLOT + NX * XSLOT;
  // Gate/up halves moved as one 3-D box {32 columns, 32 rows, 2 halves}: one TMA operation
  // instead of two for the saved Z read by the SwiGLU backward, its output e, and the Z that
  // the SwiGLU forward saves.  In shared memory the box is the two 32 x 32 staging blocks of
  // the halves, one after the other, each swizzled as a 2-D block.
  static constexpr bool PAIR_SIDE = EPI == EPI_SWIGLU_BWD;
  static constexpr bool PAIR_OUT = EPI == EPI_SWIGLU_BWD;
  static constexpr bool PAIR_AUX = EPI == EPI_SWIGLU && AUX;
  // side inputs are prefetched NSS chunks ahead (one staging set per chunk in flight); the
  // SwiGLU backward, with two side inputs and two outputs per chunk, goes deeper, except with
  // NVFP4 operands, whose larger stages leave the shared memory for two
  static constexpr int NSS0 = (EPI == EPI_SWIGLU_BWD && (KIND != KIND_NVFP4 || UN == 128)) ? 4 : 2;
  // (NSS itself is chosen below, with the pipeline stages: one chunk ahead where that is what
  // buys three two-row stages)
  // NVFP4: four scale warps write the block scales into TMEM (see the kernel)
  static constexpr int SF_WARPS = FP4 ? 4 : 0;
  // NVFP4 SwiGLU with NVFP4 output: the scale warps also form half of each tile's output
  static constexpr bool EARLY = FP4 && DUAL && OUT_DT == DT_E2M1;
  static constexpr int OUT_WARPS = NUM_EPI_WARPS + (EARLY ? SF_WARPS : 0);   // warps storing output
  static constexpr int THREADS = NUM_THREADS + 32 * SF_WARPS;
  static constexpr int BAR_BYTES = FP4 ? 384 : 320;   // barriers, then 12 bytes of flags (see the kernel)
  static constexpr int MAX_STAGES = FP4 ? 8 : 6;
  // Wide stores: OW chunks of 32 columns leave in one TMA store (a staging row of up to 128
  // bytes), so that a warp issues fewer bulk-tensor operations per tile; the number of small
  // TMA operations, not their bytes, is what competes with the mainloop's loads.  The staging
  // sets stay double-buffered: a program whose wider sets would cost a pipeline stage keeps
  // one chunk per store (measured: a single reused set made the SwiGLU backward 2% slower).
  static constexpr int OW_MAX = (OUT_DT == DT_E2M1 || NO == 0 || OUT_DT == DT_F32)
                                    ? 1
                                    : (NX > 0 ? 2 : 128 / (32 * dt_bytes(OUT_DT)));
  static constexpr int SMEM_FREE = MAX_SMEM - 1024 - BAR_BYTES;   // for the stages and the epilogue
  // Pipeline stages of sb bytes that fit beside the epilogue's staging (with the store width
  // chosen below for that stage size).
  static constexpr int stages_with(int sb, int osets = 2, int nss = NSS0) {
    const int side = nss * NS * SSLOT;
    const int narrow = fit_stages(SMEM_FREE - OUT_WARPS * (side + osets * OUTSET), sb, MAX_STAGES);
    int ow = 1;
    for (int w = 4; w >= 2; w /= 2) {
      if (ow == 1 && w <= OW_MAX && NCHUNK % w == 0 &&
          fit_stages(SMEM_FREE - OUT_WARPS * (side + osets * w * OUTSET), sb, MAX_STAGES) >= narrow)
        ow = w;
    }
    return fit_stages(SMEM_FREE - OUT_WARPS * (side + osets * ow * OUTSET), sb, MAX_STAGES);
  }
  // bf16 and e4m3 operands take two K rows per stage (64 KB stages) where three such stages
  // fit: the same bytes in flight as six stages of one row, with half the barrier round trips
  // per byte.  A K-major operand's second row is a second 128-byte-swizzled block of 128 rows;
  // an MN-major atom simply holds twice the rows of K.  Measured: the gate/up GEMM of the block
  // forward 5.6% faster, the down GEMM 4.6%, the block backward 2.3%; with two stages, G1 13%
  // slower, so it keeps one row.
  static constexpr bool KROWS2_OK = !FP4 && KIND != KIND_TF32;
  // A program whose epilogue staging leaves room for only two such stages gives up first the
  // second output staging set (waiting for each store to leave shared memory before the next:
  // G1, with its second output, 98.9 -> 95.9 us), then the side-input prefetch depth (one chunk
  // ahead: the SwiGLU and RMSNorm backward GEMMs, the block backward 2.117 -> 2.060 ms).  The
  // three-stage two-row pipeline is worth more to them than the deeper epilogue buffers.
  static constexpr int CFG = !KROWS2_OK ? 0 : stages_with(2 * SB1) >= 3 ? 1 : stages_with(2 * SB1, 1) >= 3 ? 2
                             : (NS > 0 && stages_with(2 * SB1, 1, 1) >= 3) ? 3 : 0;
  static constexpr int KROWS = CFG > 0 ? 2 : 1;
  static constexpr int OSETS = CFG >= 2 ? 1 : 2;   // output staging sets
  static constexpr int NSS = CFG == 3 ? 1 : NSS0;
  static_assert(NCHUNK % NSS == 0, "a chunk and the next tile's chunk NCHUNK later share a ring slot");
  static constexpr int SIDE_BYTES = NSS * NS * SSLOT;
  static_assert(!EARLY || OSETS == 2, "the NVFP4 SwiGLU output alternates two staging sets");
  static constexpr int A_BYTES = A_STAGE_BYTES * KROWS;          // this CTA's A in a stage
  static constexpr int B_STAGE_BYTES = B_ROW_BYTES * KROWS;
  static constexpr int STAGE_BYTES = KROWS * SB1;
  static constexpr int BK = FP4 ? 2 * BK_BYTES : KROWS * BK_BYTES / OP_BYTES;   // K elements per stage
  static constexpr int K_COORD = FP4 ? BK_BYTES : BK;   // TMA K step per stage (NVFP4 maps count bytes)
  static constexpr int S_NARROW =
      fit_stages(SMEM_FREE - OUT_WARPS * (SIDE_BYTES + OSETS * OUTSET), STAGE_BYTES, MAX_STAGES);   // one chunk per store
  static constexpr bool fits_ow(int ow) {
    return ow <= OW_MAX && NCHUNK % ow == 0 &&
           fit_stages(SMEM_FREE - OUT_WARPS * (SIDE_BYTES + OSETS * ow * OUTSET), STAGE_BYTES, MAX_STAGES) >= S_NARROW;
  }
  static constexpr int OW = fits_ow(4) ? 4 : fits_ow(2) ? 2 : 1;
  static constexpr int OUTSET_W = OW * OUTSET;               // one staging set: OW chunks of each output
  static constexpr int RB_OUT = OW * 32 * dt_bytes(OUT_DT);  // staging row bytes of the main output
  static constexpr int RB_X = OW * 64;                       // ... of the bf16 aux output
  static_assert(OW == 1 || (RB_OUT <= 128 && (NX == 0 || RB_X <= 128) && NCHUNK % OW == 0), "wide store rows");
  static constexpr int EPI_WARP_BYTES = SIDE_BYTES + OSETS * OUTSET_W;
  static constexpr int EPI_BYTES = OUT_WARPS * EPI_WARP_BYTES;
  static constexpr int STAGES = fit_stages(SMEM_FREE - EPI_BYTES, STAGE_BYTES, MAX_STAGES);
  // TMEM: two accumulators of UN columns, then (NVFP4) each stage's block scales, 4 columns
  // per atom
  static constexpr int SF_COLS = (SF_A_BYTES + SF_B_BYTES) / 128;
  static constexpr int ACC = (FP4 && UN == 256) ? 1 : 2;   // accumulators in TMEM
  static_assert(ACC * UN + STAGES * SF_COLS <= TMEM_COLS, "TMEM columns");
  static_assert(UN % 128 == 0 && UN <= UMMA_N && B_ROWS % B_BOX == 0, "MMA N");
  static_assert(!FP4 || (!A_MN && !B_MN && !AUX && (UN == 256 || UN == 128) && CG == 2),
                "NVFP4: K-major operands, CTA pairs, MMA N 256 or 128");
  // a SwiGLU tile's B rows come from two places (gate and up), one 128-row scale atom each
  static_assert(!(FP4 && DUAL) || UN == 256, "NVFP4 SwiGLU: MMA N 256");
  static_assert(OUT_DT != DT_E2M1 || (FP4 && EPI == EPI_SWIGLU), "e2m1 output: NVFP4 SwiGLU");
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
  static_assert(STAGES >= 2, "shared memory budget");
  // barriers: full and empty per stage, 2 + 2 accumulator, side loads, done; NVFP4 adds per
  // stage the scales-landed (this CTA) and scales-in-TMEM (leader) barriers
  static constexpr int NBAR = 2 * STAGES + 5 + NSS * NUM_EPI_WARPS + (FP4 ? 2 * STAGES : 0);
  static_assert(8 * NBAR + 12 <= BAR_BYTES, "barrier area");
  static_assert(!(A_MN || B_MN) || KIND != KIND_TF32, "MN-major operands are bf16 or e4m3");
  // MN-major operands: a 128-byte swizzle row holds MN_ATOM elements of M (or N); one atom is
  // BK rows of K; a 128-row tile is BM / MN_ATOM atoms; one MMA consumes UMMA_K rows of K
  static constexpr int MN_ATOM = 128 / OP_BYTES;
  static constexpr int MN_ATOM_BYTES = BK * 128;
  static constexpr int UMMA_K = 32 / OP_BYTES;
  static_assert(!AUX || EPI == EPI_SWIGLU || EPI == EPI_RESID, "aux output: SwiGLU or residual programs");
  static_assert(CG == 1 || CG == 2, "CTA group");
  // instruction descriptor: D f32, A/B format, operand majors, N >> 3, M >> 4.  Block-scaled
  // (NVFP4): bits 4-5 and 29-30 select the scale columns' byte (0: all four used by a 4X
  // vector), the formats are e2m1 (1), bit 23 = 0 selects ue4m3 scales, and D is f32.
  static constexpr uint32_t FMT = KIND == KIND_BF16 ? 1u : KIND == KIND_TF32 ? 2u : KIND == KIND_NVFP4 ? 1u : 0u;
  static constexpr uint32_t IDESC = (FP4 ? 0u : 1u << 4) | (FMT << 7) | (FMT << 10) | ((A_MN ? 1u : 0u) << 15) |
                                    ((B_MN ? 1u : 0u) << 16) | ((uint32_t)(UN >> 3) << 17) |
                                    ((uint32_t)(PAIR_ROWS >> 4) << 24);
};

// Shared-memory matrix descriptor, 128B swizzle, version 1 (sm_100 family).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Tile order.  Tiles come in groups of group_n consecutive N-tiles; inside a group the
// N-tile index runs fastest, then the M-tile.  The CTAs working at the same time then share
// a few A row-blocks and one group's slice of B, which stays resident in L2 while the group
// sweeps all M-tiles.
__device__ __forceinline__ void tile_coords(int tile, const GemmParams& p, int& mb, int& nb) {
  const int per_group = p.m_tiles * p.group_n;
  const int g = tile / per_group;
  const int n_first = g * p.group_n;
  const int gsize = min(p.group_n, p.n_tiles - n_first);
  const int t = tile - g * per_group;
  mb = t / gsize;
  nb = n_first + (t - mb * gsize);
}

// Work item w -> (tile coordinates, K slice).  The K slice is the slowest index, so the CTAs
// working at the same time share one slice of K.
__device__ __forceinline__ void work_coords(int w, const GemmParams& p, int& mb, int& nb, int& kb0, int& kb1,
                                            int num_kb) {
  const int tiles = p.m_tiles * p.n_tiles;
  const int ks = w / tiles;
  tile_coords(w - ks * tiles, p, mb, nb);
  kb0 = ks * p.kb_per_split;
  kb1 = min(num_kb, kb0 + p.kb_per_split);
}

struct Watch {
  volatile int* abort;
  int* status;
  uint64_t timeout_ns;
};

// Bounded wait on an mbarrier phase.  False = gave up (timeout here, or abort elsewhere).
__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, const Watch& w, int site) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*w.abort) return false;
    if (ptx::globaltimer() - t0 > w.timeout_ns) {
      *w.abort = 1;
      __threadfence_block();
      if (w.status) atomicCAS(w.status, 0, site);
      return false;
    }
  }
}
// Short bounded wait used only while draining after an abort (never raises anything).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > 20000000ull) return;
  }
}

// ------------------------------------------------------- swizzled 32 x 32 staging blocks
// A staging block holds 32 rows of 32 elements; row bytes RB = 32 * elem size; 16-byte
// chunk j of row i sits at chunk j ^ ((i * RB / 128) & (RB / 16 - 1)), which is the TMA
// 32/64/128-byte swizzle for that row width.  Thread i touches row i only; the XOR spreads
// 8 consecutive rows over all 32 banks.
// The same for staging rows of RB bytes (32 <= RB <= 128, a wide store's block): 16-byte unit
// u of row i sits at u ^ ((i * RB / 128) & (RB / 16 - 1)).
template <int RB>
__device__ __forceinline__ uint32_t swz_rb(uint32_t slot, int row, int u) {
  constexpr int MASK = RB / 16 - 1;
  return slot + row * RB + ((u ^ ((row * RB >> 7) & MASK)) << 4);
}
template <int DT>
__device__ __forceinline__ uint32_t swz(uint32_t slot, int row, int j) {
  return swz_rb<32 * dt_bytes(DT)>(slot, row, j);
}

template <int DT>
__device__ __forceinline__ void slot_read(uint32_t slot, int row, float (&x)[32]) {
  if constexpr (DT == DT_BF16) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 u = ptx::ld_shared_v4(swz<DT>(slot, row, j));
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        x[8 * j + 2 * k] = __uint_as_float(w[k] << 16);
        x[8 * j + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
      }
    }
  } else if constexpr (DT == DT_F32) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint4 u = ptx::ld_shared_v4(swz<DT>(slot, row, j));
      x[4 * j] = __uint_as_float(u.x);
      x[4 * j + 1] = __uint_as_float(u.y);
      x[4 * j + 2] = __uint_as_float(u.z);
      x[4 * j + 3] = __uint_as_float(u.w);
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&b);
}
__device__ __forceinline__ float round_bf16(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// Writes the 32 values of a chunk into row `row` of a staging block whose rows are RB bytes,
// starting at 16-byte unit u0 of the row (a wide block holds several chunks side by side).
template <int DT, int RB = 32 * dt_bytes(DT)>
__device__ __forceinline__ void slot_write(uint32_t slot, int row, const float (&x)[32], int u0 = 0) {
  if constexpr (DT == DT_BF16) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      ptx::st_shared_v4(swz_rb<RB>(slot, row, u0 + j), pack_bf16(x[8 * j], x[8 * j + 1]),
                        pack_bf16(x[8 * j + 2], x[8 * j + 3]), pack_bf16(x[8 * j + 4], x[8 * j + 5]),
                        pack_bf16(x[8 * j + 6], x[8 * j + 7]));
  } else if constexpr (DT == DT_F32) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      ptx::st_shared_v4(swz_rb<RB>(slot, row, u0 + j), __float_as_uint(x[4 * j]), __float_as_uint(x[4 * j + 1]),
                        __float_as_uint(x[4 * j + 2]), __float_as_uint(x[4 * j + 3]));
  } else {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int e = 16 * j + 4 * k;
        w[k] = (uint32_t)ptx::cvt_e4m3x2(x[e], x[e + 1]) | ((uint32_t)ptx::cvt_e4m3x2(x[e + 2], x[e + 3]) << 16);
      }
      ptx::st_shared_v4(swz_rb<RB>(slot, row, u0 + j), w[0], w[1], w[2], w[3]);
    }
  }
}

// An e4m3 chunk from codes already packed in pairs (q[i] holds elements 2i, 2i+1), into a
// staging block with rows of RB bytes from unit u0 on.
template <int RB = 32>
__device__ __forceinline__ void slot_write_codes(uint32_t slot, int row, const uint16_t (&q)[16], int u0 = 0) {
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) w[k] = (uint32_t)q[8 * j + 2 * k] | ((uint32_t)q[8 * j + 2 * k + 1] << 16);
    ptx::st_shared_v4(swz_rb<RB>(slot, row, u0 + j), w[0], w[1], w[2], w[3]);
  }
}

// Value as it will be stored (used where a partial must match the stored tensor).
template <int DT>
__device__ __forceinline__ float as_stored(float x) {
  if constexpr (DT == DT_BF16) return round_bf16(x);
  else return x;
}

// Lane l returns sum over the 32 lanes of x[l] (x is consumed).  31 shuffles.
__device__ __forceinline__ float warp_transpose_sum(float (&x)[32], int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? x[i] : x[i + off];
      const float keep = upper ? x[i + off] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return x[0];
}

__device__ __forceinline__ float silu_f(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

// NVFP4 quantisation of one block of 16 values with tensor scale s: sf = e4m3(amax / (6 s)),
// q = e2m1(x * (1 / (sf s))) (all zero when sf is 0), each product, quotient and reciprocal
// rounded once in fp32.  q[0..1] receive the 16 codes (element 2j in the low nibble of byte j);
// returns the scale's e4m3 byte.  The quantiser kernel and the SwiGLU epilogue both decide
// through here.
__device__ __forceinline__ uint32_t nvfp4_block16(const float* x, float s, uint32_t* q) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(x[j]));
  const float u = __fdiv_rn(amax, __fmul_rn(6.0f, s));
  const uint16_t code2 = ptx::cvt_e4m3x2(u, 0.0f);   // low byte: e4m3(u), saturating at 448
  float sfv, zero;
  ptx::e4m3x2_to_f32(code2, sfv, zero);
  const float d = __fmul_rn(sfv, s);
  const float rd = d > 0.f ? __frcp_rn(d) : 0.f;
  float y[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) y[j] = __fmul_rn(x[j], rd);
  q[0] = ptx::cvt_e2m1x8(y);
  q[1] = ptx::cvt_e2m1x8(y + 8);
  return code2 & 0xFFu;
}
__device__ __forceinline__ float sigmoid_f(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// =====================================================================================
template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    gemm_epilogue_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ CUtensorMap tmSide0,
                         const __grid_constant__ CUtensorMap tmSide1, const __grid_constant__ CUtensorMap tmAux,
                         const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                         const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t sm_stage = base;
  const uint32_t sm_epi = base + C::STAGES * C::STAGE_BYTES;
  const uint32_t sm_bar = sm_epi + C::EPI_BYTES;
  const int NBAR = C::NBAR;
  uint8_t* misc = smem_raw + (sm_bar - raw) + 8 * NBAR;
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  // CTA pairs: the second CTA's producer leaves its k-block count here, in the leader, for the
  // leader's drain at exit (bit 31: it dropped its first k-block, the test hook)
  volatile uint32_t* peer_iters = reinterpret_cast<volatile uint32_t*>(misc + 8);

#define FULL_BAR(s) (sm_bar + 8u * (s))
#define EMPTY_BAR(s) (sm_bar + 8u * (C::STAGES + (s)))
#define TFULL_BAR(a) (sm_bar + 8u * (2 * C::STAGES + (a)))
#define TEMPTY_BAR(a) (sm_bar + 8u * (2 * C::STAGES + 2 + (a)))
#define SIDE_BAR(w, s) (sm_bar + 8u * (2 * C::STAGES + 4 + C::NSS * (w) + (s)))
#define DONE_BAR (sm_bar + 8u * (2 * C::STAGES + 4 + C::NSS * NUM_EPI_WARPS))
#define SFULL_BAR(s) (sm_bar + 8u * (2 * C::STAGES + 5 + C::NSS * NUM_EPI_WARPS + (s)))
#define SREADY_BAR(s) (sm_bar + 8u * (3 * C::STAGES + 5 + C::NSS * NUM_EPI_WARPS + (s)))

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = C::CG == 2 ? ptx::cluster_ctarank() : 0u;   // position in the CTA pair
  const bool leader = rank == 0;
  const int cluster_id = blockIdx.x / C::CG, n_clusters = gridDim.x / C::CG;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(FULL_BAR(s), 1);
      ptx::mbar_init(EMPTY_BAR(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(TFULL_BAR(a), 1);
      ptx::mbar_init(TEMPTY_BAR(a), C::OUT_WARPS * C::CG);   // every warp of the pair that reads it
    }
    for (int w = 0; w < NUM_EPI_WARPS; ++w)
      for (int s = 0; s < C::NSS; ++s) ptx::mbar_init(SIDE_BAR(w, s), 1);
    ptx::mbar_init(DONE_BAR, 1);
    if constexpr (C::FP4) {
      for (int s = 0; s < C::STAGES; ++s) {
        ptx::mbar_init(SFULL_BAR(s), 1);                  // this CTA's producer + scale bytes
        ptx::mbar_init(SREADY_BAR(s), C::SF_WARPS * C::CG);   // every scale warp of the pair
      }
    }
    *abort_flag = 0;
    *peer_iters = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    if constexpr (C::FP4) {
      ptx::prefetch_tmap(&tmSFA);
      ptx::prefetch_tmap(&tmSFB);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc<C::CG>(ptx::smem_u32(const_cast<uint32_t*>(tmem_holder)), TMEM_COLS);
    ptx::tmem_relinquish<C::CG>();
  }
  ptx::tc_fence_before();
  if constexpr (C::CG == 2)
    ptx::cluster_sync();   // the peer's barriers are initialised before any remote arrive
  else
    __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // Stream order.  Everything above touched only this CTA's shared memory and TMEM.  The
  // epilogue waits for the previous kernel before its first global access (side inputs, row
  // and column vectors, stores).  With F_AB_READY the caller guarantees that the previous
  // kernel writes neither A nor B (all earlier work is complete once that kernel has started,
  // see griddep_launch_dependents), so the producer streams them at once and the MMA warp,
  // which touches no global memory, does not wait.
  if (!(p.flags & F_AB_READY) || warp >= 2) {
    ptx::griddep_wait();
    ptx::griddep_launch_dependents();
  }

  const Watch watch{abort_flag, p.status, p.timeout_ns};
  const int total_tiles = p.m_tiles * p.n_tiles * p.k_splits;   // work items
  // Producer (warp 0, lane 0): k-blocks it went through (issued, or dropped by the test hook)
  // and whether it dropped the first one.  Its copies of k-block i land on FULL_BAR(i %
  // STAGES) in phase i / STAGES; at exit these counts tell which phases may still be open.
  int prod_iters = 0;
  bool prod_skip0 = false;
  const int num_kb = (p.K + C::BK - 1) / C::BK;

  // NVFP4 SwiGLU output with its one accumulator: a quarter's epilogue warp and scale warp split
  // each tile, NCHUNK / 2 chunks of 32 output columns each.  Each reads its chunks' gate and up
  // halves from TMEM, hands TMEM back at once (one arrival per warp), then forms, quantises and
  // stores the outputs while the next tile's MMAs run; `between` runs after each chunk's store.
  auto early_half = [&](uint32_t tacc, int c0, int n0, int r0, float sc, uint32_t out_base, uint64_t pol,
                        float& amax_local, auto&& between) {
    constexpr int NH = C::NCHUNK / 2;
    const int row = r0 + lane;
    uint32_t gv[NH][32], uv[NH][32];
#pragma unroll
    for (int c = 0; c < NH; ++c) {
      ptx::tmem_ld32(tacc + 32 * (c0 + c), gv[c]);
      ptx::tmem_ld32(tacc + C::UN / 2 + 32 * (c0 + c), uv[c]);
    }
    ptx::tmem_ld_wait();
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa(TEMPTY_BAR(0), 0));
    // The arithmetic stays below the hand-back: the values pass through an empty volatile asm,
    // which keeps its place after the arrival (without it the compiler moved the SwiGLU above
    // the arrival, where it held the accumulator).
#pragma unroll
    for (int c = 0; c < NH; ++c)
#pragma unroll
      for (int j = 0; j < 32; ++j) asm volatile("" : "+r"(gv[c][j]), "+r"(uv[c][j]));
    float abuf[NH][32];
#pragma unroll
    for (int c = 0; c < NH; ++c) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float G = __uint_as_float(gv[c][j]) * sc, U = __uint_as_float(uv[c][j]) * sc;
        const float a = silu_f(G) * U;
        amax_local = fmaxf(amax_local, fabsf(a));
        abuf[c][j] = a;
      }
    }
#pragma unroll
    for (int c = 0; c < NH; ++c) {
      const int col0 = n0 + 32 * (c0 + c);
      uint32_t q4[4];
      const uint32_t sfc =
          nvfp4_block16(abuf[c], p.fp4_scale, q4) | (nvfp4_block16(abuf[c] + 16, p.fp4_scale, q4 + 2) << 8);
      if (row < p.M && col0 < p.N)
        *reinterpret_cast<uint16_t*>(p.out_sf + sf_offset(row, col0 / 16, p.out_sf_kc)) = (uint16_t)sfc;
      const uint32_t oslot = out_base + (c & 1) * C::OUTSET;
      if (lane == 0) ptx::bulk_wait_read<1>();  // the group that last used this set is done reading
      __syncwarp();
      ptx::st_shared_v4(oslot + 16 * lane, q4[0], q4[1], q4[2], q4[3]);   // 32 rows of 16 bytes
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (col0 < p.N && r0 < p.M) ptx::tma_store_2d_hint(&tmOut, col0 / 2, r0, oslot, pol);
        ptx::bulk_commit();
      }
      between();
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool skip = (p.flags & F_INJECT_SKIP) || ((p.flags & F_INJECT_RANK0) && rank == 0) ||
                  ((p.flags & F_INJECT_RANK1) && rank == 1);
      prod_skip0 = skip;
      bool ok = true;
      const uint64_t keep = ptx::make_policy_evict_last();   // B: reused by every M-tile of a group
      const uint64_t normal =
          (p.flags & F_A_STREAM) ? ptx::make_policy_evict_first() : ptx::make_policy_evict_normal();
      for (int tile = cluster_id; ok && tile < total_tiles; tile += n_clusters) {
        int mb, nb, kb0, kb1;
        work_coords(tile, p, mb, nb, kb0, kb1, num_kb);
        const int m0 = mb * C::PAIR_ROWS + (int)rank * BM;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!bwait(EMPTY_BAR(stage), phase ^ 1u, watch, SITE_PRODUCER_EMPTY)) {
            ok = false;
            break;
          }
          if (skip) {
            skip = false;  // test hook: this k-block never arrives
          } else {
            const uint32_t fb = FULL_BAR(stage);
            const uint32_t sa = sm_stage + stage * C::STAGE_BYTES;
            const uint32_t sb = sa + C::A_BYTES;
            const int k0 = kb * C::K_COORD;
            // the leader's full barrier counts the operand bytes of both CTAs of a pair
            if (leader) ptx::mbar_arrive_expect_tx(fb, C::CG * (C::A_BYTES + C::B_STAGE_BYTES));
            auto load = [&](uint32_t dst, const CUtensorMap* m, int c0, int c1, uint64_t pol) {
              if constexpr (C::CG == 2)
                ptx::tma_load_2d_pair(dst, m, c0, c1, ptx::mapa(fb, 0), pol);
              else
                ptx::tma_load_2d_hint(dst, m, c0, c1, fb, pol);
            };
            if constexpr (C::A_MN) {
#pragma unroll
              for (int j = 0; j < BM / C::MN_ATOM; ++j)
                load(sa + C::MN_ATOM_BYTES * j, &tmA, m0 + C::MN_ATOM * j, k0, normal);
            } else {   // KROWS rows of K, each its own 128-byte-swizzled block of 128 rows
#pragma unroll
              for (int a = 0; a < C::KROWS; ++a)
                load(sa + a * A_STAGE_BYTES, &tmA, k0 + a * (BK_BYTES / C::OP_BYTES), m0, normal);
            }
            // B: this CTA's B_ROWS rows of the tile's UN (SwiGLU: UN / 2 gate rows, then up rows)
            if constexpr (C::B_MN) {
              const int n0 = nb * C::UN + (int)rank * C::B_ROWS;
#pragma unroll
              for (int j = 0; j < C::B_ROWS / C::MN_ATOM; ++j)
                load(sb + C::MN_ATOM_BYTES * j, &tmB, n0 + C::MN_ATOM * j, k0, keep);
            } else {
              constexpr int HALF = C::UN / 2;
#pragma unroll
              for (int h = 0; h < C::B_ROWS / C::B_BOX; ++h) {
                const int off = ((int)rank * (C::B_ROWS / C::B_BOX) + h) * C::B_BOX;   // row offset in the tile
                const int row = C::DUAL ? (off < HALF ? nb * HALF + off : p.up_offset + nb * HALF + off - HALF)
                                        : nb * C::UN + off;
#pragma unroll
                for (int a = 0; a < C::KROWS; ++a)
                  load(sb + a * C::B_ROW_BYTES + C::B_BOX * BK_BYTES * h, &tmB, k0 + a * (BK_BYTES / C::OP_BYTES), row,
                       keep);
              }
            }
            if constexpr (C::FP4) {
              // block scales: KSTEPS atoms (one per MMA) for this CTA's A rows, then for each 128
              // rows of the tile's N (SwiGLU: the gate rows' block, then the up rows'); an atom
              // row of the maps is one 512-byte atom.  They land on this CTA's own barrier,
              // which its scale warps wait on.
              const uint32_t ssf = sb + C::B_STAGE_BYTES;
              const uint32_t sfb_bar = SFULL_BAR(stage);
              const int kc = p.K / 64;
              ptx::mbar_arrive_expect_tx(sfb_bar, C::SF_A_BYTES + C::SF_B_BYTES);
              ptx::tma_load_2d_hint(ssf, &tmSFA, 0, (m0 / 128) * kc + KSTEPS * kb, sfb_bar, normal);
#pragma unroll
              for (int j = 0; j < C::UN / 128; ++j) {
                const int blk = C::DUAL ? (j == 0 ? nb : p.up_offset / 128 + nb) : nb * (C::UN / 128) + j;
                ptx::tma_load_2d_hint(ssf + C::SF_A_BYTES + KSTEPS * 512 * j, &tmSFB, 0, blk * kc + KSTEPS * kb,
                                      sfb_bar, keep);
              }
            }
          }
          ++prod_iters;
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Let this CTA's copies still in flight land before it exits (at once when every phase
      // has completed, the normal case).  A k-block older than the last STAGES was consumed by
      // the MMA, so its phase is complete.  A pair's operand copies complete on the leader's
      // barriers, which only the leader can poll: the leader drains them for both CTAs at exit.
      for (int i = max(0, prod_iters - C::STAGES); i < prod_iters; ++i) {
        if (prod_skip0 && i == 0) continue;
        if constexpr (C::CG == 1) drain_wait(FULL_BAR(i % C::STAGES), (uint32_t)(i / C::STAGES) & 1u);
        if constexpr (C::FP4) drain_wait(SFULL_BAR(i % C::STAGES), (uint32_t)(i / C::STAGES) & 1u);
      }
      if constexpr (C::CG == 2) {
        if (rank != 0)
          ptx::st_cluster_u32(ptx::mapa(ptx::smem_u32(const_cast<uint32_t*>(peer_iters)), 0),
                              (uint32_t)prod_iters | (prod_skip0 ? 0x80000000u : 0u));
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {   // the pair's MMAs are issued by its leader CTA
      int stage = 0;
      uint32_t phase = 0;
      int t = 0;
      bool ok = true;
      for (int tile = cluster_id; ok && tile < total_tiles; tile += n_clusters, ++t) {
        const int acc = t % C::ACC;
        const uint32_t aph = (t / C::ACC) & 1;
        if (!bwait(TEMPTY_BAR(acc), aph ^ 1u, watch, SITE_MMA_TMEM_EMPTY)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * C::UN;
        int mb_, nb_, kb0, kb1;
        work_coords(tile, p, mb_, nb_, kb0, kb1, num_kb);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!bwait(FULL_BAR(stage), phase, watch, SITE_MMA_FULL)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = sm_stage + stage * C::STAGE_BYTES;
          const uint32_t sb = sa + C::A_BYTES;
          if constexpr (C::FP4) {
            // the scale warps of both CTAs have written this stage's block scales into TMEM
            // (A: 4 columns per MMA; B: 4 per MMA and 128 rows of N)
            if (!bwait(SREADY_BAR(stage), phase, watch, SITE_MMA_SCALES)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint32_t tsa = tmem_base + C::ACC * C::UN + stage * C::SF_COLS;
            const uint32_t tsb = tsa + 4 * KSTEPS;
            constexpr int NB128 = C::UN / 128;
#pragma unroll
            for (int k = 0; k < KSTEPS; ++k) {
              const uint64_t ad = smem_desc(sa + k * 32, 16, 1024);
              const uint64_t bd = smem_desc(sb + k * 32, 16, 1024);
              ptx::umma_nvfp4<C::CG>(d_tmem, ad, bd, C::IDESC, tsa + 4 * k, tsb + 4 * NB128 * k,
                                     (kb != kb0 || k != 0) ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int k = 0; k < KSTEPS * C::KROWS; ++k) {
              const int kr = k / KSTEPS, ks = k % KSTEPS;   // row of K in the stage, 32-byte step in it
              const uint64_t ad = C::A_MN ? smem_desc(sa + k * C::UMMA_K * 128, C::MN_ATOM_BYTES, 1024)
                                          : smem_desc(sa + kr * A_STAGE_BYTES + ks * 32, 16, 1024);
              const uint64_t bd = C::B_MN ? smem_desc(sb + k * C::UMMA_K * 128, C::MN_ATOM_BYTES, 1024)
                                          : smem_desc(sb + kr * C::B_ROW_BYTES + ks * 32, 16, 1024);
              ptx::umma<C::KIND, C::CG>(d_tmem, ad, bd, C::IDESC, (kb != kb0 || k != 0) ? 1u : 0u);
            }
          }
          ptx::umma_commit<C::CG>(EMPTY_BAR(stage));  // frees the stage (in both CTAs) once done
          if (++stage == C::STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::umma_commit<C::CG>(TFULL_BAR(acc));  // accumulator complete (both CTAs)
      }
      // every MMA (and the arrivals its commits make) is complete before TMEM is released
      ptx::umma_commit<C::CG>(DONE_BAR, 1);
      drain_wait(DONE_BAR, 0);
    }
    __syncwarp();
  } else if (warp < 2 + NUM_EPI_WARPS) {
    // ------------------------------------------------------------ epilogue warps
    const int ew = warp - 2;  // staging ownership
    const int q = warp & 3;   // TMEM lane quadrant this warp may read
    const uint32_t side_base = sm_epi + ew * C::EPI_WARP_BYTES;
    const uint32_t out_base = side_base + C::NSS * C::NS * C::SSLOT;
    uint32_t side_par = 0, side_pending = 0;
    uint32_t prefetched = 0;   // chunks (< NSS) of the coming tile whose side inputs are in flight
    float amax_local = 0.f;
    const uint64_t stream_pol = ptx::make_policy_evict_first();  // outputs and side inputs: touched once
    bool ok = true;
    int t = 0;
    for (int tile = cluster_id; ok && tile < total_tiles; tile += n_clusters, ++t) {
      int mb, nb, kb0_, kb1_;
      work_coords(tile, p, mb, nb, kb0_, kb1_, num_kb);
      const int m0 = mb * C::PAIR_ROWS + (int)rank * BM;
      const int n0 = nb * C::BN_OUT;
      const int r0 = m0 + 32 * q;   // first row of this warp's 32-row slab
      const int row = r0 + lane;
      const bool row_ok = row < p.M;
      const int acc = t % C::ACC;
      const uint32_t aph = (t / C::ACC) & 1;

      // A chunk is live if some of its rows and columns are in range; side loads of dead
      // chunks are neither issued nor waited for.
      const bool slab_ok = r0 < p.M;
      auto live = [&](int c) { return slab_ok && (n0 + 32 * c < p.N); };
      // side inputs of chunk c of the tile at (tn0, tr0) into ring slot c % NSS
      auto issue_side_at = [&](int c, int tn0, int tr0) {
        if constexpr (C::NS > 0) {
          const int slot = c % C::NSS;
          const uint32_t sbar = SIDE_BAR(ew, slot);
          const uint32_t dst = side_base + slot * C::NS * C::SSLOT;
          const bool side1 = C::NS > 1 && !(p.flags & F_NO_SIDE1);
          ptx::mbar_arrive_expect_tx(sbar, (side1 ? C::NS : 1) * C::SSLOT);
          if constexpr (C::EPI == EPI_RESID) {
            ptx::tma_load_2d_hint(dst, &tmSide0, tn0 + 32 * c, tr0, sbar, stream_pol);
          } else if constexpr (C::PAIR_SIDE) {
            ptx::tma_load_3d_hint(dst, &tmSide0, tn0 + 32 * c, tr0, 0, sbar, stream_pol);   // G and U blocks
          } else {
            ptx::tma_load_2d_hint(dst, &tmSide0, tn0 + 32 * c, tr0, sbar, stream_pol);
            if (side1) ptx::tma_load_2d_hint(dst + C::SSLOT, &tmSide1, tn0 + 32 * c, tr0, sbar, stream_pol);
          }
        }
      };
      // The next tile of this CTA: its first chunks' side inputs are issued while this tile's
      // last chunks are processed, so its epilogue does not start on a cold load.
      const int next_tile = tile + n_clusters;
      int nn0 = 0, nr0 = 0;
      bool next_slab_ok = false;
      if constexpr (C::NS > 0) {
        if (next_tile < total_tiles) {
          int nmb, nnb, nk0, nk1;
          work_coords(next_tile, p, nmb, nnb, nk0, nk1, num_kb);
          nn0 = nnb * C::BN_OUT;
          nr0 = nmb * C::PAIR_ROWS + (int)rank * BM + 32 * q;
          next_slab_ok = nr0 < p.M;
        }
      }
      auto live_next = [&](int c) { return next_slab_ok && (nn0 + 32 * c < p.N); };
      if constexpr (C::NS > 0) {
#pragma unroll
        for (int c = 0; c < C::NSS; ++c) {
          if (c < C::NCHUNK && live(c) && !((prefetched >> c) & 1u)) {
            if (lane == 0) issue_side_at(c, n0, r0);
            side_pending |= 1u << c;
          }
        }
        prefetched = 0;
      }

      float rs = 1.f, rc = 0.f;
      if ((p.flags & F_ROWSCALE) && row_ok) rs = __ldg(p.row_scale + row);
      if constexpr (C::EPI == EPI_RMSBWD || C::EPI == EPI_XENT_BWD) {
        if (row_ok) rc = __ldg(p.row_coef + row);   // c (RMSNorm backward) or lse (cross-entropy)
      }
      int target = -1;
      if constexpr (C::EPI == EPI_XENT || C::EPI == EPI_XENT_BWD) {
        if (row_ok) target = __ldg(p.row_index + row);
      }
      float xmax = -INFINITY, xsum = 0.f, xtgt = 0.f;   // online softmax state of this row's tile
      const float ts = p.tensor_scale;

      // RoPE: the rotation table entries of a chunk (16 pairs of this row's position) are
      // loaded a chunk ahead, the first chunk's before the accumulator is waited for
      constexpr bool ROPE = C::EPI == EPI_ROPE;
      float4 rcv[ROPE ? 4 : 1], rsv[ROPE ? 4 : 1];
      auto rope_fetch = [&](int c) {
        if constexpr (ROPE) {
          const int col = n0 + 32 * c;
          if (col < p.rope_ncols) {
            const int pos = row % p.rope_seq_len;
            const size_t base = (size_t)pos * (p.rope_head_dim >> 1) + ((col % p.rope_head_dim) >> 1);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              rcv[j] = __ldg(reinterpret_cast<const float4*>(p.rope_cos + base) + j);
              rsv[j] = __ldg(reinterpret_cast<const float4*>(p.rope_sin + base) + j);
            }
          }
        }
      };
      rope_fetch(0);
      ok = bwait(TFULL_BAR(acc), aph, watch, SITE_EPI_TMEM_FULL);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t tacc = tmem_base + ((uint32_t)(32 * q) << 16) + acc * C::UN;
      float rowacc = 0.f;

      // NVFP4 SwiGLU output: this warp forms the first half of the tile (the scale warp of the
      // same TMEM lane quarter, the second half)
      constexpr bool EARLY = C::EARLY;
      if constexpr (EARLY) early_half(tacc, 0, n0, r0, ts * rs, out_base, stream_pol, amax_local, [] {});

#pragma unroll 1
      for (int c = 0; c < (EARLY ? 0 : C::NCHUNK); ++c) {
        float x[32];
        float xu[C::DUAL ? 32 : 1];
        {
          uint32_t v[32];
          ptx::tmem_ld32(tacc + 32 * c, v);
          if constexpr (C::DUAL) {
            uint32_t u[32];
            ptx::tmem_ld32(tacc + C::UN / 2 + 32 * c, u);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) xu[j] = __uint_as_float(u[j]);
          } else {
            ptx::tmem_ld_wait();
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]);
        }
        if (c == C::NCHUNK - 1) {  // accumulator fully read: hand it back to the (leader's) MMA warp
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if constexpr (C::CG == 2)
              ptx::mbar_arrive_cluster(ptx::mapa(TEMPTY_BAR(acc), 0));
            else
              ptx::mbar_arrive(TEMPTY_BAR(acc));
          }
        }

        // side inputs of this chunk
        float s0[C::NS > 0 ? 32 : 1];
        float s1[C::NS > 1 ? 32 : 1];
        if constexpr (C::NS > 0) {
          const int slot = c % C::NSS;
          if (live(c)) {
            bool sok = bwait(SIDE_BAR(ew, slot), (side_par >> slot) & 1u, watch, SITE_EPI_SIDE);
            sok = __all_sync(0xffffffffu, sok);
            if (!sok) {
              ok = false;
              break;
            }
            side_par ^= 1u << slot;
            side_pending &= ~(1u << slot);
            const uint32_t src = side_base + slot * C::NS * C::SSLOT;
            slot_read<C::SIDE_DT>(src, lane, s0);
            if constexpr (C::NS > 1) {
              if (p.flags & F_NO_SIDE1) {
#pragma unroll
                for (int j = 0; j < 32; ++j) s1[j] = 0.f;
              } else {
                slot_read<C::SIDE_DT>(src + C::SSLOT, lane, s1);
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              s0[j] = 0.f;
              if constexpr (C::NS > 1) s1[j] = 0.f;
            }
          }
          __syncwarp();
          if (c + C::NSS < C::NCHUNK) {
            if (live(c + C::NSS)) {
              if (lane == 0) issue_side_at(c + C::NSS, n0, r0);
              side_pending |= 1u << slot;
            }
          } else if (live_next(c + C::NSS - C::NCHUNK)) {   // same slot: NCHUNK is a multiple of NSS
            if (lane == 0) issue_side_at(c + C::NSS - C::NCHUNK, nn0, nr0);
            side_pending |= 1u << slot;
            prefetched |= 1u << (c + C::NSS - C::NCHUNK);
          }
        }

        const int col0 = n0 + 32 * c;
        float o1[C::NO > 1 ? 32 : 1];
        constexpr bool CODES = C::EPI == EPI_SWIGLU_BWD && C::OUT_DT == DT_E4M3;   // e quantised in place
        uint16_t qg[CODES ? 16 : 1], qu[CODES ? 16 : 1];
        constexpr bool FP4_OUT = C::OUT_DT == DT_E2M1;   // NVFP4 codes + block scales of the SwiGLU output
        uint32_t q4[FP4_OUT ? 4 : 1];
        uint32_t sfc = 0;
        float zg[C::AUX ? 32 : 1], zu[C::NX > 1 ? 32 : 1];

        // ---------------------------------------------------------------- the program
        if constexpr (C::EPI == EPI_STORE) {
          if (p.flags & F_COLSCALE) {
            const float4* g4 = reinterpret_cast<const float4*>(p.col_scale + col0);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 g = __ldg(g4 + j);
              x[4 * j] *= ts * g.x;
              x[4 * j + 1] *= ts * g.y;
              x[4 * j + 2] *= ts * g.z;
              x[4 * j + 3] *= ts * g.w;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] *= ts;
          }
        } else if constexpr (C::EPI == EPI_RESID) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            x[j] = fmaf(x[j], ts, s0[j]);
            const float st = as_stored<C::OUT_DT>(x[j]);
            rowacc = fmaf(st, st, rowacc);
          }
          if constexpr (C::AUX) {   // u = h * g, the column vector broadcast along the tile
            const float4* g4 = reinterpret_cast<const float4*>(p.col_scale + col0);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 g = __ldg(g4 + j);
              zg[4 * j] = x[4 * j] * g.x;
              zg[4 * j + 1] = x[4 * j + 1] * g.y;
              zg[4 * j + 2] = x[4 * j + 2] * g.z;
              zg[4 * j + 3] = x[4 * j + 3] * g.w;
            }
          }
        } else if constexpr (C::EPI == EPI_ROWSCALE) {
          const float sc = ts * rs;
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] *= sc;
        } else if constexpr (C::EPI == EPI_SWIGLU) {
          const float sc = ts * rs;
          const float os = p.out_scale;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float G = x[j] * sc, U = xu[j] * sc;
            if constexpr (C::AUX) {
              zg[j] = G;
              zu[j] = U;
            }
            const float a = silu_f(G) * U;
            amax_local = fmaxf(amax_local, fabsf(a));
            x[j] = a * os;
          }
          if constexpr (FP4_OUT) {   // two blocks of 16 columns (os is 1 here)
            sfc = nvfp4_block16(x, p.fp4_scale, q4) | (nvfp4_block16(x + 16, p.fp4_scale, q4 + 2) << 8);
            if (row_ok && col0 < p.N)
              *reinterpret_cast<uint16_t*>(p.out_sf + sf_offset(row, col0 / 16, p.out_sf_kc)) = (uint16_t)sfc;
          }
        } else if constexpr (C::EPI == EPI_ROPE) {
          const float sc = ts * rs;
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] *= sc;
          if (col0 < p.rope_ncols) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float4 cv = rcv[j], sv = rsv[j];
              const float cs[4] = {cv.x, cv.y, cv.z, cv.w};
              const float sn[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int e = 8 * j + 2 * k;
                const float a0 = x[e], a1 = x[e + 1];
                x[e] = a0 * cs[k] - a1 * sn[k];
                x[e + 1] = a0 * sn[k] + a1 * cs[k];
              }
            }
          }
          if (c + 1 < C::NCHUNK) rope_fetch(c + 1);
        } else if constexpr (C::EPI == EPI_SWIGLU_BWD) {
          const float sc = ts * rs;
          if constexpr (C::OUT_DT == DT_E4M3) {
            // e is quantised once: its e4m3 codes (of e * os) go to the staging blocks as they
            // are, and the partial sums the dequantised values (scaled back once per row below)
            const float os = p.out_scale;
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              float eg[2], eu[2];
#pragma unroll
              for (int k = 0; k < 2; ++k) {
                const float G = s0[j + k], U = s1[j + k], d = sc * x[j + k];
                const float sg = sigmoid_f(G);
                eg[k] = d * U * sg * (1.f + G * (1.f - sg));
                eu[k] = d * G * sg;
                amax_local = fmaxf(amax_local, fmaxf(fabsf(eg[k]), fabsf(eu[k])));
              }
              qg[j >> 1] = ptx::cvt_e4m3x2(eg[0] * os, eg[1] * os);
              qu[j >> 1] = ptx::cvt_e4m3x2(eu[0] * os, eu[1] * os);
              float g0, g1, u0, u1;
              ptx::e4m3x2_to_f32(qg[j >> 1], g0, g1);
              ptx::e4m3x2_to_f32(qu[j >> 1], u0, u1);
              rowacc = fmaf(g0, s0[j], fmaf(u0, s1[j], fmaf(g1, s0[j + 1], fmaf(u1, s1[j + 1], rowacc))));
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float G = s0[j], U = s1[j], d = sc * x[j];
              const float sg = sigmoid_f(G);
              const float eg = as_stored<C::OUT_DT>(d * U * sg * (1.f + G * (1.f - sg)));
              const float eu = as_stored<C::OUT_DT>(d * G * sg);
              rowacc = fmaf(eg, G, fmaf(eu, U, rowacc));
              x[j] = eg;
              o1[j] = eu;
            }
          }
        } else if constexpr (C::EPI == EPI_XENT) {
          // P4 / P5: block log-sum-exp with the running (max, sum-exp) state of the row
          const float sc = ts * rs;
          float cm = -INFINITY;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            x[j] = (col0 + j < p.N) ? x[j] * sc : -INFINITY;
            cm = fmaxf(cm, x[j]);
          }
          if (cm > xmax) {
            xsum *= __expf(xmax - cm);
            xmax = cm;
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            xsum += (x[j] == -INFINITY) ? 0.f : __expf(x[j] - xmax);   // out-of-range columns add nothing
            if (col0 + j == target) xtgt = x[j];
          }
        } else if constexpr (C::EPI == EPI_XENT_BWD) {
          const float sc = ts * rs;
          const float gs = rs * p.out_scale;   // r * dloss / M
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const bool in = col0 + j < p.N;
            const float z = x[j] * sc;
            const float pj = in ? __expf(z - rc) : 0.f;
            const float e = as_stored<C::OUT_DT>(gs * (pj - (col0 + j == target ? 1.f : 0.f)));
            rowacc = in ? fmaf(e, z, rowacc) : rowacc;
            x[j] = e;
          }
        } else if constexpr (C::EPI == EPI_RMSBWD) {
          float ht[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            x[j] *= ts;                 // t
            ht[j] = s0[j] * x[j];       // h * t
          }
          if (p.flags & F_COLSCALE) {
            const float4* g4 = reinterpret_cast<const float4*>(p.col_scale + col0);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float4 g = __ldg(g4 + j);
              const float gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) x[4 * j + k] *= gv[k];
            }
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) x[j] = x[j] - rc * s0[j] + s1[j];
          if (p.flags & F_COLPART) {
            const float colsum = warp_transpose_sum(ht, lane);
            if (slab_ok && col0 + lane < p.N) p.col_part[(size_t)(r0 >> 5) * p.col_part_ld + col0 + lane] = colsum;
          }
        }

        // ---------------------------------------------------------------- stage + store
        // OW chunks form one store group: their blocks sit side by side in wide staging rows
        // and leave in one TMA store per output after the group's last chunk.
        if constexpr (C::NO == 0) continue;
        constexpr int OW = C::OW;
        constexpr int OBLK = OW * C::OSLOT;             // one output block of a staging set
        constexpr int XBLK = OW * C::XSLOT;             // one aux block
        constexpr int UO = 2 * dt_bytes(C::OUT_DT);     // 16-byte units of a chunk's output row
        const int h = c % OW;                           // the chunk's place in its group
        const uint32_t oset = out_base + ((c / OW) % C::OSETS) * C::OUTSET_W;
        if (h == 0) {
          if (lane == 0) ptx::bulk_wait_read<C::OSETS - 1>();  // the group that last used this set is read
          __syncwarp();
        }
        if constexpr (FP4_OUT) {
          ptx::st_shared_v4(oset + 16 * lane, q4[0], q4[1], q4[2], q4[3]);   // 32 rows of 16 bytes (OW = 1)
        } else if constexpr (CODES) {
          slot_write_codes<C::RB_OUT>(oset, lane, qg, h * UO);
          slot_write_codes<C::RB_OUT>(oset + OBLK, lane, qu, h * UO);
        } else {
          slot_write<C::OUT_DT, C::RB_OUT>(oset, lane, x, h * UO);
          if constexpr (C::NO > 1) slot_write<C::OUT_DT, C::RB_OUT>(oset + OBLK, lane, o1, h * UO);
        }
        if constexpr (C::NX > 0) slot_write<DT_BF16, C::RB_X>(oset + C::NO * OBLK, lane, zg, h * 4);
        if constexpr (C::NX > 1) slot_write<DT_BF16, C::RB_X>(oset + C::NO * OBLK + XBLK, lane, zu, h * 4);
        if (h == OW - 1) {
          const int gcol = col0 - 32 * (OW - 1);        // first column of the group
          const bool store = gcol < p.N && r0 < p.M;
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (store) {
              if constexpr (C::PAIR_OUT) {
                ptx::tma_store_3d_hint(&tmOut, gcol, r0, 0, oset, stream_pol);   // e's gate and up blocks
              } else if (C::EPI == EPI_STORE && C::OUT_DT == DT_F32 && p.k_splits > 1) {
                ptx::tma_reduce_add_2d_hint(&tmOut, gcol, r0, oset, stream_pol);   // split-K partial
              } else {
                ptx::tma_store_2d_hint(&tmOut, FP4_OUT ? gcol / 2 : gcol, r0, oset, stream_pol);
              }
              if constexpr (C::PAIR_AUX) {
                ptx::tma_store_3d_hint(&tmAux, gcol, r0, 0, oset + C::NO * OBLK, stream_pol);   // Z's G and U
              } else if constexpr (C::NX > 0) {
                ptx::tma_store_2d_hint(&tmAux, gcol, r0, oset + C::NO * OBLK, stream_pol);
              }
            }
            ptx::bulk_commit();
          }
        }
      }
      if (!ok) break;
      if constexpr (C::EPI == EPI_SWIGLU_BWD && C::OUT_DT == DT_E4M3) rowacc *= 1.f / p.out_scale;
      if constexpr (C::EPI == EPI_RESID || C::EPI == EPI_SWIGLU_BWD || C::EPI == EPI_XENT_BWD) {
        if ((C::EPI != EPI_RESID || (p.flags & F_PARTIAL)) && row_ok)
          p.row_part[(size_t)nb * p.row_part_ld + row] = rowacc;
      }
      if constexpr (C::EPI == EPI_XENT) {
        if (row_ok) {
          p.row_part[(size_t)nb * p.row_part_ld + row] = xmax;
          p.row_part2[(size_t)nb * p.row_part_ld + row] = xsum;
          if (target >= n0 && target < n0 + C::BN_OUT) p.row_out[row] = xtgt;
        }
      }
    }
    if constexpr (C::EPI == EPI_SWIGLU || (C::EPI == EPI_SWIGLU_BWD && C::OUT_DT == DT_E4M3)) {
      if (p.flags & F_AMAX) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
          amax_local = fmaxf(amax_local, __shfl_xor_sync(0xffffffffu, amax_local, off));
        if (lane == 0 && amax_local > 0.f) atomicMax(p.amax, __float_as_uint(amax_local));
      }
    }
    if (lane == 0) {
      ptx::bulk_wait<0>();  // every TMA store of this warp has completed
      if (!ok) {
        for (int s = 0; s < C::NSS; ++s)
          if (side_pending & (1u << s)) drain_wait(SIDE_BAR(ew, s), (side_par >> s) & 1u);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ scale warps (NVFP4)
    // Warp w writes TMEM lane quarter w % 4 of this CTA.  The block-scaled MMA reads row m of
    // A's scales from lane m, column base + m / 32 of each 4-column group, and every quarter
    // reads all 256 rows of B's scales from its own lanes (row n: lane n % 32 of the quarter,
    // column 4 (n / 128) + (n % 128) / 32 of each 8-column group).  So per stage, once its
    // scales have landed in this CTA's shared memory, each warp stores A's scales of its 32 rows
    // into the one column per MMA read for them, and B's scales into the 8 columns per MMA:
    // stores from registers run beside the MMAs, where copies into TMEM would stall them.
    if constexpr (C::FP4) {
      const uint32_t q = (uint32_t)(warp & 3);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      // cursor over this CTA's k-blocks, in the MMA's order, whose scales go to TMEM next
      int s_tile = cluster_id, s_kb = 0, s_kb1 = 0;
      auto s_enter = [&]() {
        if (s_tile < total_tiles) {
          int mb_, nb_;
          work_coords(s_tile, p, mb_, nb_, s_kb, s_kb1, num_kb);
        }
      };
      s_enter();
      int staged = 0;   // k-blocks whose scales are in TMEM
      auto stage_scales = [&]() {
        if (!__all_sync(0xffffffffu, bwait(SFULL_BAR(stage), phase, watch, SITE_SCALES_FULL))) return false;
        // atom row `lane` of a scale atom holds rows lane + 32 i (i = 0..3), 4 scales each
        const uint32_t ssf = sm_stage + stage * C::STAGE_BYTES + C::A_BYTES + C::B_STAGE_BYTES + 16 * lane;
        const uint32_t tcol = tmem_base + ((32u * q) << 16) + C::ACC * C::UN + stage * C::SF_COLS;
#pragma unroll
        for (int k = 0; k < KSTEPS; ++k)
          ptx::tmem_st_x1(tcol + 4 * k + q, ptx::ld_shared_u32(ssf + 512 * k + 4 * q));
#pragma unroll
        for (int k = 0; k < KSTEPS; ++k) {
          if constexpr (C::UN == 256)
            ptx::tmem_st_x8(tcol + 4 * KSTEPS + 8 * k, ptx::ld_shared_v4(ssf + C::SF_A_BYTES + 512 * k),
                            ptx::ld_shared_v4(ssf + C::SF_A_BYTES + KSTEPS * 512 + 512 * k));
          else   // MMA N 128: one atom of B rows, 4 columns per MMA
            ptx::tmem_st_x4(tcol + 4 * KSTEPS + 4 * k, ptx::ld_shared_v4(ssf + C::SF_A_BYTES + 512 * k));
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa(SREADY_BAR(stage), 0));
        if (++stage == C::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        if (++s_kb == s_kb1) {
          s_tile += n_clusters;
          s_enter();
        }
        ++staged;
        return true;
      };
      if constexpr (!C::EARLY) {
        while (ok && s_tile < total_tiles) ok = stage_scales();
      } else {
        // Also the second half of each tile's NVFP4 SwiGLU output.  Before waiting for a tile's
        // accumulator, the scales of the tile and of the next tile's first two stages go to TMEM,
        // so that the next tile's MMAs start as soon as both halves have handed TMEM back; after
        // each of this warp's output chunks, the next stages whose scales have landed follow
        // (without waiting), and the rest of the ring after the tile.  (Staging the whole ring
        // first held the hand-back until its loads had landed: 0.80 ms for the 8B gate/up GEMM,
        // against 0.75 with two stages and 0.72 with the stages staged between chunks.)
        const uint32_t out_base = sm_epi + (NUM_EPI_WARPS + (warp - 2 - NUM_EPI_WARPS)) * C::EPI_WARP_BYTES;
        const uint64_t stream_pol = ptx::make_policy_evict_first();
        float amax_local = 0.f;
        int through = 0;   // k-blocks of the tiles up to this one
        int t = 0;
        for (int tile = cluster_id; ok && tile < total_tiles; tile += n_clusters, ++t) {
          int mb, nb, kb0, kb1;
          work_coords(tile, p, mb, nb, kb0, kb1, num_kb);
          through += kb1 - kb0;
          int ahead = 0, ahead_full = 0;
          if (tile + n_clusters < total_tiles) {
            int mb2, nb2, k0, k1;
            work_coords(tile + n_clusters, p, mb2, nb2, k0, k1, num_kb);
            ahead_full = min(C::STAGES, k1 - k0);
            ahead = min(2, ahead_full);
          }
          while (ok && staged < through + ahead) ok = stage_scales();
          if (!ok) break;
          const int r0 = mb * C::PAIR_ROWS + (int)rank * BM + 32 * (int)q;
          const int row = r0 + lane;
          const float rs = ((p.flags & F_ROWSCALE) && row < p.M) ? __ldg(p.row_scale + row) : 1.f;
          ok = __all_sync(0xffffffffu, bwait(TFULL_BAR(0), (uint32_t)(t & 1), watch, SITE_EPI_TMEM_FULL));
          if (!ok) break;
          ptx::tc_fence_after();
          early_half(tmem_base + ((32u * q) << 16), C::NCHUNK / 2, nb * C::BN_OUT, r0, p.tensor_scale * rs, out_base,
                     stream_pol, amax_local, [&] {
                       while (ok && staged < through + ahead_full &&
                              __all_sync(0xffffffffu, ptx::mbar_test_wait(SFULL_BAR(stage), phase)))
                         ok = stage_scales();
                     });
        }
        if (p.flags & F_AMAX) {
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1)
            amax_local = fmaxf(amax_local, __shfl_xor_sync(0xffffffffu, amax_local, off));
          if (lane == 0 && amax_local > 0.f) atomicMax(p.amax, __float_as_uint(amax_local));
        }
        if (lane == 0) ptx::bulk_wait<0>();   // every TMA store of this warp has completed
      }
    }
    __syncwarp();
  }

  if constexpr (C::CG == 2) {
    // Both CTAs' operand copies of a k-block complete on the leader's full barrier, in one
    // phase that the leader arms (arrive + expect_tx of both CTAs' bytes).  After an abort
    // the two producers may have gone through different numbers of k-blocks, leaving phases
    // that can never complete on their own: armed by the leader with bytes the second CTA
    // never sent, or receiving the second CTA's bytes without being armed.  Once every role
    // of both CTAs has stopped (this barrier; it also makes the second CTA's count visible),
    // the leader completes those phases for the missing side and waits, bounded, until every
    // copy has landed.  Only then does the pair meet at the final barrier below, after which
    // either CTA may exit.
    ptx::tc_fence_before();
    ptx::cluster_sync();
    if (warp == 0 && lane == 0 && leader) {
      const uint32_t w = *peer_iters;
      const int n_l = prod_iters, n_p = (int)(w & 0x7FFFFFFFu);
      const bool skip_l = prod_skip0, skip_p = (w >> 31) != 0;
      constexpr uint32_t PEER_BYTES = C::A_BYTES + C::B_STAGE_BYTES;
      for (int i = max(0, min(n_l, n_p) - C::STAGES); i < max(n_l, n_p); ++i) {
        const bool by_l = i < n_l && !(skip_l && i == 0);
        const bool by_p = i < n_p && !(skip_p && i == 0);
        if (!by_l && !by_p) continue;
        const uint32_t fb = FULL_BAR(i % C::STAGES);
        if (by_l && !by_p) ptx::mbar_complete_tx(fb, PEER_BYTES);       // bytes that will never come
        if (!by_l && by_p) ptx::mbar_arrive_expect_tx(fb, PEER_BYTES);  // arm it for the bytes that do
        drain_wait(fb, (uint32_t)(i / C::STAGES) & 1u);
      }
    }
  }
  ptx::tc_fence_before();
  if constexpr (C::CG == 2)
    ptx::cluster_sync();   // no remote arrive or load still targets this CTA's memory
  else
    __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc<C::CG>(tmem_base, TMEM_COLS);
  }
#undef FULL_BAR
#undef EMPTY_BAR
#undef TFULL_BAR
#undef TEMPTY_BAR
#undef SIDE_BAR
#undef DONE_BAR
#undef SFULL_BAR
#undef SREADY_BAR
}

// ------------------------------------------------------------------ host launcher
struct GemmLaunch {
  CUtensorMap tmA, tmB, tmOut, tmSide0, tmSide1, tmAux;
  CUtensorMap tmSFA, tmSFB;   // NVFP4 block scales of A and B (unused otherwise)
  GemmParams p;
  int sms;
  int overlap;   // launch with a programmatic dependency on the previous kernel of the stream
};

using GemmLaunchFn = cudaError_t (*)(const GemmLaunch&, cudaStream_t);

// Number of CTA groups (pairs for CG = 2) that can be resident at once, per device.
template <class C>
int resident_groups(int sms) {
  static std::atomic<int> cached[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int n = sms / C::CG;
  if constexpr (C::CG == 2) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, gemm_epilogue_kernel<C>, &cfg) == cudaSuccess && clusters > 0)
      n = clusters < n ? clusters : n;
    cudaGetLastError();
  }
  if (dev < 64) cached[dev] = n;
  return n;
}

template <class C>
cudaError_t launch_gemm(const GemmLaunch& L, cudaStream_t s) {
  static std::atomic<int> attr_done[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(gemm_epilogue_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done[dev] = 1;
  }
  // persistent grid: one CTA group per resident slot, at most one per work item
  const int64_t tiles = (int64_t)L.p.m_tiles * L.p.n_tiles * L.p.k_splits;
  const int groups = (int)(tiles < resident_groups<C>(L.sms) ? tiles : resident_groups<C>(L.sms));
  if (groups <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int na = 0;
  if constexpr (C::CG == 2) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 2;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (L.overlap) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.gridDim = dim3(C::CG * groups, 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, gemm_epilogue_kernel<C>, L.tmA, L.tmB, L.tmOut, L.tmSide0, L.tmSide1, L.tmAux,
                            L.tmSFA, L.tmSFB, L.p);
}

}  // namespace coda
