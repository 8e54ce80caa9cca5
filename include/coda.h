/*
 * coda.h — C ABI of the GB300 (sm_103a) GEMM-epilogue library (libcoda.so).
 *
 * What the library computes.  A GEMM whose output tile stays on chip while a short
 * "epilogue program" runs on it before the single store to HBM; and the Transformer
 * block chains built from such GEMMs, chiefly the reparameterised
 * GEMM -> residual -> RMSNorm -> GEMM chain, in which the first GEMM emits per-row
 * partial sums of squares, a light reduce turns them into the RMS scale r, and the second
 * GEMM applies r per row because a per-row scalar commutes with the matmul.
 *
 * Sources (page title, section):
 *   [KuCoin]     "CODA: new research optimizes Transformer training with GEMM-epilogue
 *                programming" (kucoin.com news flash):
 *                "CODA: «El epílogo» esconde un tesoro" (mainloop / epilogue split, the
 *                deferred-r rewrite, partial RMS + light reduce, backward inherits the
 *                structure), "Cinco «bloques» y un «lenguaje LEGO»" (the five epilogue
 *                primitive kinds), "hoja de referencia" (coverage: RMSNorm, residual,
 *                SwiGLU, RoPE, cross-entropy and their gradients; single GPU).
 *   [Ecosistema] "CODA: Nuevo kernel GPU reduce costos de entrenamiento IA"
 *                (ecosistemastartup.com), "¿Qué es GEMM-epilogue…?" (C = alpha*A*B + beta*C;
 *                epilogue = scaling, bias, activation, residual add, precision cast).
 *
 * Conventions for every call.
 *   - Memory: the caller owns every buffer.  Tensor pointers are DEVICE pointers on the
 *     current CUDA device.  The library allocates no device memory in any call.  An output
 *     must not overlap any input or other output of the same call, unless the call says so
 *     (the chains start a GEMM before the previous kernel ends when that kernel writes none of
 *     the GEMM's operands, which relies on it).
 *   - Streams: every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream) and does not synchronise, except
 *     coda_get_device_status, whose name says it reads the device.
 *   - Errors: every call returns an int status (CODA_OK = 0 or a negative CODA_ERR_*).
 *     Arguments are checked on the host before anything is launched; a rejected call has
 *     launched nothing.  A wait inside a kernel that runs out of time (see
 *     coda_set_watchdog_ms) ends that kernel early with wrong output and sets the device
 *     status word, read by coda_get_device_status.
 *   - Layout: a coda_tensor is a logical [rows, cols] matrix.  CODA_ROW_MAJOR stores
 *     element (i, j) at ptr[i*ld + j]; CODA_COL_MAJOR at ptr[j*ld + i].  `ptr` must be
 *     16-byte aligned and ld * element size a multiple of 16 bytes (CODA_ERR_ALIGN).
 *   - Precision: bf16 and e4m3 operands, fp32 accumulation in tensor memory, one rounding
 *     at the store; fp32 operands run on the tensor cores as tf32.
 *   - Hardware: sm_103a (GB300) only.  Calls on any other device return CODA_ERR_NO_DEVICE.
 */
#ifndef CODA_H_
#define CODA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CODA_API __attribute__((visibility("default")))
#else
#define CODA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ status codes */
enum coda_status {
  CODA_OK = 0,
  CODA_ERR_NULL = -1,                /* a required pointer is NULL */
  CODA_ERR_SHAPE = -2,               /* inconsistent or unsupported sizes */
  CODA_ERR_ALIGN = -3,               /* base or leading dimension not 16-byte aligned */
  CODA_ERR_DTYPE = -4,               /* unsupported dtype combination */
  CODA_ERR_UNSUPPORTED_PROGRAM = -5, /* op list with no compiled epilogue */
  CODA_ERR_LAUNCH = -6,              /* CUDA launch / descriptor encoding failed */
  CODA_ERR_DEVICE_TIMEOUT = -7,      /* a kernel wait ran out of time (device status) */
  CODA_ERR_NO_DEVICE = -8            /* no sm_103 device current, or driver entry missing */
};

/* CODA_NVFP4: e2m1 codes packed two per byte along the row (element 2j in the low nibble of
 * byte j); rows, cols and ld count elements (cols and ld even, ld / 2 bytes a multiple of 16),
 * ROW_MAJOR only.  Each row carries one e4m3 block scale per 16 consecutive elements, kept
 * apart in the block-scale layout described at coda_quantize_nvfp4, and the tensor carries an
 * fp32 scale s: element value = s * block scale * code value.  The pages name FP4 only as a
 * format that speeds up the matmul [KuCoin, "El «impuesto a la pereza» para entrenar modelos
 * grandes"]; the block size 16 with e4m3 scales is the NVFP4 format of the tensor cores. */
enum coda_dtype { CODA_F32 = 0, CODA_BF16 = 1, CODA_E4M3 = 2, CODA_NVFP4 = 3 };
enum coda_layout { CODA_ROW_MAJOR = 0, CODA_COL_MAJOR = 1 };

typedef struct coda_tensor {
  void* ptr;      /* device pointer, 16-byte aligned */
  int32_t dtype;  /* enum coda_dtype */
  int32_t layout; /* enum coda_layout */
  int64_t rows;   /* logical rows */
  int64_t cols;   /* logical columns */
  int64_t ld;     /* leading dimension in elements (stride of the outer storage index) */
} coda_tensor;

/* ------------------------------------------------------------- epilogue programs
 * An epilogue program is an ordered list of ops applied to the fp32 accumulator tile
 * acc = A . W^T before the store.  Op kinds follow the five primitive kinds of
 * [KuCoin, "Cinco bloques y un lenguaje LEGO"]: elementwise / pairwise transforms,
 * vector loads (row or column vectors), matrix-block loads / stores (side inputs, saved
 * activations), block reductions (partials), state (running amax).  The list must match
 * one of the compiled programs below, else CODA_ERR_UNSUPPORTED_PROGRAM:
 *
 *   {}                                        out = acc
 *   {COL_SCALE}                               out = acc * g[j]
 *   {TENSOR_SCALE}                            out = s * acc
 *   {[TENSOR_SCALE,] ADD_SIDE [, ROW_SUMSQ_PARTIAL] [, STORE_COL_SCALED]}
 *        out = s * acc + R; partials of out^2; STORE_COL_SCALED also stores
 *        out * g[j] (the RMSNorm gain broadcast along the tile) to aux.store_aux
 *   {ROW_SCALE}                               out = r[i] * acc
 *   {[TENSOR_SCALE,] ROW_SCALE, [STORE_AUX,] SWIGLU [, AMAX]}
 *        W holds 2N rows (gate rows [0, N), up rows [N, 2N)); Z = s * r[i] * acc over
 *        2N columns; out = silu(Z_gate) * Z_up (times out_scale); STORE_AUX saves Z.
 *   {ROW_SCALE, ROPE}                         out = rope(r[i] * acc)
 *   {SWIGLU_BWD, ROW_SCALE, ROW_DOT_PARTIAL [, AMAX]}   (optionally TENSOR_SCALE first)
 *        dA = s * acc; with Z = [G | U] from aux_in:
 *        out[:, j] = r dA U silu'(G),  out[:, N + j] = r dA silu(G)   (out is [M, 2N]);
 *        row partials of sum_j out . Z.  e4m3 out: the codes of out * out_scale are stored,
 *        the partials sum the dequantised values (code / out_scale) and AMAX keeps max |out|
 *        before quantisation.
 *   {[TENSOR_SCALE,] RMSBWD_COMBINE [, COL_DOT_PARTIAL]}   t = s * acc; h = aux_in, dY =
 *        aux_in2 (optional), g = side.col_scale (optional, 1 when NULL):
 *        out = g[j] t - c[i] h [+ dY]; COL_DOT_PARTIAL (needs g): column partials of h * t
 *   {[TENSOR_SCALE,] [ROW_SCALE,] XENT_PARTIAL}    z = s * r[i] * acc are logits (never stored;
 *        out only gives the shape [M, V], its ptr may be NULL); per 256-column tile t and row i:
 *        aux.row_partials[t, i] = max_j z_ij, aux.row_partials2[t, i] = sum_j exp(z_ij - max),
 *        and aux.row_values[i] = z[i, side.row_index[i]] (the target's logit)
 *   {[TENSOR_SCALE,] [ROW_SCALE,] XENT_BWD, ROW_DOT_PARTIAL}   z as above, lse = side.row_coef:
 *        out = r[i] * out_scale * (exp(z - lse_i) - [j == side.row_index[i]]); row partials of
 *        sum_j out * z
 */
enum coda_op {
  CODA_OP_TENSOR_SCALE = 1,      /* acc *= side.tensor_scale */
  CODA_OP_ROW_SCALE = 2,         /* acc[i, :] *= side.row_scale[i] */
  CODA_OP_COL_SCALE = 3,         /* acc[:, j] *= side.col_scale[j] */
  CODA_OP_ADD_SIDE = 4,          /* acc += side.residual[i, j] */
  CODA_OP_SWIGLU = 5,            /* gate/up halves -> silu(gate) * up */
  CODA_OP_ROPE = 6,              /* rotate adjacent pairs of the first rope_ncols columns */
  CODA_OP_SWIGLU_BWD = 7,        /* SwiGLU backward (see above) */
  CODA_OP_RMSBWD_COMBINE = 8,    /* RMSNorm backward combine (see above) */
  CODA_OP_ROW_SUMSQ_PARTIAL = 9, /* aux.row_partials[t, i] = sum over tile t of out^2 */
  CODA_OP_ROW_DOT_PARTIAL = 10,  /* aux.row_partials[t, i] = sum over tile t of out . Z */
  CODA_OP_COL_DOT_PARTIAL = 11,  /* aux.col_partials[b, j] = sum over 32-row block b of h * t */
  CODA_OP_AMAX = 12,             /* atomic max of |out| before the e4m3 cast into *aux.amax */
  CODA_OP_STORE_AUX = 13,        /* save the pre-activation Z to aux.store_aux */
  CODA_OP_STORE_COL_SCALED = 14, /* also store out[i, j] * side.col_scale[j] to aux.store_aux [M, N] bf16 */
  CODA_OP_XENT_PARTIAL = 15,     /* online (max, sum-exp) state and target logit per row and tile */
  CODA_OP_XENT_BWD = 16          /* softmax-minus-onehot gradient of the cross-entropy */
};

#define CODA_MAX_OPS 8
typedef struct coda_epilogue_program {
  int32_t n_ops;
  int32_t ops[CODA_MAX_OPS];
} coda_epilogue_program;

typedef struct coda_side_inputs {
  const coda_tensor* residual;  /* ADD_SIDE: [M, N], ROW_MAJOR, dtype of out (bf16/f32) */
  const float* row_scale;       /* ROW_SCALE: r [M] */
  const float* row_coef;        /* RMSBWD_COMBINE: c [M] */
  const float* col_scale;       /* COL_SCALE, RMSBWD_COMBINE: g [N], 16-byte aligned */
  const coda_tensor* aux_in;    /* SWIGLU_BWD: Z [M, 2N] bf16; RMSBWD_COMBINE: h [M, N] bf16 */
  const coda_tensor* aux_in2;   /* RMSBWD_COMBINE: dY [M, N] bf16 */
  const float* rope_cos;        /* ROPE: [rope_seq_len, rope_head_dim / 2] fp32 */
  const float* rope_sin;        /* ROPE: same shape */
  int32_t rope_seq_len;         /* ROPE: position of row i is i mod rope_seq_len */
  int32_t rope_head_dim;        /* ROPE: 32, 64, 128 or 256 */
  int32_t rope_ncols;           /* ROPE: columns [0, rope_ncols) rotated; multiple of head_dim */
  float tensor_scale;           /* TENSOR_SCALE: s (e.g. s_x * s_w for fp8) */
  float out_scale;              /* e4m3 outputs: 1 / scale before the cast (> 0); XENT_BWD: dloss / M */
  const int32_t* row_index;     /* XENT_PARTIAL, XENT_BWD: [M] target class of each row, in [0, N) */
  const void* a_block_scales;   /* NVFP4 A: its block scales (16-byte aligned) */
  const void* w_block_scales;   /* NVFP4 W: its block scales (16-byte aligned) */
  float out_fp4_scale;          /* NVFP4 out: the tensor scale s of the stored codes (> 0) */
} coda_side_inputs;

typedef struct coda_aux_outputs {
  float* row_partials;          /* [ceil(N / 256), row_partials_ld] (SWIGLU_BWD: tiles of dA) */
  int64_t row_partials_ld;      /* >= M */
  float* col_partials;          /* [ceil(M / 32), col_partials_ld]: one row per 32-row slab */
  int64_t col_partials_ld;      /* >= N */
  const coda_tensor* store_aux; /* STORE_AUX: Z [M, 2N] bf16; STORE_COL_SCALED: [M, N] bf16 */
  float* amax;                  /* AMAX: one float; the caller zeroes it before the call */
  float* row_partials2;         /* XENT_PARTIAL: sum-exp partials, same layout as row_partials */
  float* row_values;            /* XENT_PARTIAL: [M] logit of each row's target */
  void* out_block_scales;       /* NVFP4 out: block scales of the codes (16-byte aligned) */
} coda_aux_outputs;

/* out = epilogue(prog, A . W^T): one GEMM whose fp32 tile stays on chip while the program runs
 * [KuCoin, "El epílogo esconde un tesoro" (fixed mainloop, programmable epilogue before the
 * single store); Ecosistema, "¿Qué es GEMM-epilogue…?" (C = alpha A B + beta C; scaling,
 * activation, residual add, cast in the epilogue)].
 *   A    logical [M, K]: ROW_MAJOR (K contiguous) or COL_MAJOR (M contiguous).
 *   W    logical [N, K] (nn.Linear [out, in] layout when ROW_MAJOR); [2N, K] for SWIGLU.
 *   out  logical [M, N] ROW_MAJOR ([M, 2N] for SWIGLU_BWD).
 * Operand dtypes: bf16 x bf16, e4m3 x e4m3, f32 x f32 (tf32, ROW_MAJOR only), NVFP4 x NVFP4
 * (ROW_MAJOR, K a multiple of 256, block scales in side.a_block_scales / w_block_scales, the
 * product of the tensor scales as TENSOR_SCALE; programs {}, {TENSOR_SCALE}, the ADD_SIDE
 * program, and the SWIGLU program with a bf16 or NVFP4 out; an NVFP4 out takes its tensor
 * scale from side.out_fp4_scale and writes its block scales to aux.out_block_scales); which
 * layouts each program has compiled is listed in the variant tables (others return
 * CODA_ERR_UNSUPPORTED_PROGRAM or CODA_ERR_DTYPE).  N must be a multiple of 32 (of 128 for SWIGLU), K >= 1.  M = 0 or N = 0 is a
 * no-op.  `side` and `aux` may be NULL when the program needs none of their fields. */
CODA_API int coda_gemm_epilogue(const coda_tensor* A, const coda_tensor* W, const coda_epilogue_program* prog,
                       const coda_side_inputs* side, const coda_tensor* out, const coda_aux_outputs* aux,
                       void* stream);

/* The light row reduce [KuCoin, "El epílogo esconde un tesoro"].
 *   partials: fp32 [nparts, ld] (part t of row i at partials[t*ld + i]), summed in a fixed
 *   order, so the result does not depend on the launch: up to 16 parts, part t into running sum
 *   t % 4 and then (0 + 1) + (2 + 3); above, part t into running sum t % 8 and then
 *   ((0 + 4) + (1 + 5)) + ((2 + 6) + (3 + 7)).
 *   mode CODA_REDUCE_RSQRT_MEAN: out[i] = 1 / sqrt(sum_t P[t, i] / d + eps)   (r)
 *   mode CODA_REDUCE_SCALE_SUM:  out[i] = rowscale[i] * sum_t P[t, i] / d     (c = r s / d) */
enum coda_reduce_mode { CODA_REDUCE_RSQRT_MEAN = 0, CODA_REDUCE_SCALE_SUM = 1 };
CODA_API int coda_rms_partial_reduce(const float* partials, int64_t ld, int32_t nparts, int64_t M, int64_t d, float eps,
                            int32_t mode, const float* rowscale, float* out, void* stream);

/* Full-row RMS scale: r[i] = 1 / sqrt(mean_j X[i, j]^2 + eps) for X bf16 [M, d] ROW_MAJOR
 * [KuCoin, "El epílogo esconde un tesoro" (the light reduce that yields r), here over a stored
 * activation that no GEMM epilogue produced].  r_out: fp32 [M], 16-byte aligned.  M = 0 is a
 * no-op; d < 1 returns CODA_ERR_SHAPE. */
CODA_API int coda_row_rms(const coda_tensor* X, float eps, float* r_out, void* stream);

/* [KuCoin, "Cinco bloques…" (vector load: the RMSNorm weights broadcast)]
 * RMS scale and gain broadcast in one pass over X (bf16 [M, d] ROW_MAJOR):
 *   r[i] = 1 / sqrt(mean_j X[i, j]^2 + eps),  u[i, j] = X[i, j] * g[j] (bf16 [M, d]).
 * The RMSNorm of a stored activation, split as the deferred-r chains use it. */
CODA_API int coda_rms_gain(const coda_tensor* X, const float* g, float eps, float* r_out, const coda_tensor* u_out,
                           void* stream);

/* The light reduce of the cross-entropy partials [KuCoin, "Cinco bloques…": block
 * log-sum-exp and the max / sum-exp state]: per row,
 *   lse[i] = m + log(sum_t Ps[t, i] exp(Pm[t, i] - m)),  m = max_t Pm[t, i]
 * (the tiles folded into eight running (max, scaled sum) states, tile t into state t % 8,
 * which are then merged in order: the result does not depend on the launch);
 *   loss[i] = lse[i] - target_logit[i]  (NaN when targets[i] is outside [0, V));
 *   *mean = sum_i loss[i] / M (fixed-order reduction; mean may be NULL). */
CODA_API int coda_xent_combine(const float* Pm, const float* Ps, int64_t ld, int32_t nparts, int64_t M,
                               const float* target_logit, const int32_t* targets, int64_t V, float* lse, float* loss,
                               float* mean, void* stream);

/* Column reduce [KuCoin, "El epílogo esconde un tesoro" (the backward inherits the partial +
 * light-reduce structure: here the gain gradient dg from per-slab column partials)]:
 *   out[j] = sum_b parts[b*ld + j] over b in [0, nblocks) (fixed order, so deterministic:
 *   b into running sum (b mod 32, (b / 32) mod 8) up to the last whole 256-row sweep, the rest
 *   into sum (b mod 32, 0); each group of 8 as ((0 + 1) + (2 + 3)) + ((4 + 5) + (6 + 7)), then
 *   the 32 groups in order).
 * parts: fp32 [nblocks, ld] device, ld >= N; out: fp32 [N].  N = 0 or nblocks = 0 writes
 * nothing / zeros respectively; negative sizes return CODA_ERR_SHAPE. */
CODA_API int coda_col_reduce(const float* parts, int64_t nblocks, int64_t N, int64_t ld, float* out, void* stream);

/* Gain fold [KuCoin, "Cinco bloques…" (vector load of the RMSNorm weights) and "El epílogo
 * esconde un tesoro" (the normalisation's per-column factor moved onto the next GEMM)]:
 *   W'[n, k] = W[n, k] * g[k] * (1 / out_scale)
 * The RMSNorm gain moved onto the weight of the GEMM that follows the norm, optionally
 * requantised for an FP8 GEMM.  W and W_out are ROW_MAJOR [N, K]:
 *   - bf16 -> bf16 (K a multiple of 8) or fp32 -> fp32 (K a multiple of 4): out_scale = 1 gives
 *     the plain fold; W_out may alias W.
 *   - bf16 -> e4m3 (K a multiple of 16): W_out receives the e4m3 codes of W g / out_scale
 *     (round to nearest even, saturating to +-448), so that out_scale * code is the folded
 *     weight; out_scale is its per-tensor scale (e.g. max_nk |W g| / 448).  No aliasing.
 * The product is taken in fp32 (W g, then times the fp32 reciprocal of out_scale), one rounding
 * at the store.  g: fp32 [K] device, 16-byte aligned (CODA_ERR_ALIGN).  out_scale must be
 * finite and > 0.  Other dtype pairs: CODA_ERR_DTYPE; mismatched shapes, K not a multiple of
 * the vector width, a column-major tensor or an aliased e4m3 output: CODA_ERR_SHAPE. */
CODA_API int coda_fold_gain(const coda_tensor* W, const float* g, float out_scale, const coda_tensor* W_out,
                            void* stream);

/* [KuCoin, "Cinco bloques…" (RoPE as a pairwise transform)]
 * RoPE table: cos/sin[pos, p] = cos/sin(pos * base^(-2p / head_dim)), fp32
 * [seq_len, head_dim / 2], angles evaluated in fp64 on the device. */
CODA_API int coda_rope_table(int32_t seq_len, int32_t head_dim, double base, float* cos_out, float* sin_out, void* stream);

/* ------------------------------------------------------------ block chains
 * [KuCoin, "El epílogo esconde un tesoro" (GEMM -> residual -> RMSNorm -> GEMM with partial
 * RMS, a light reduce and r deferred past the second GEMM) and "Resultados del experimento"
 * (LLaMA-style blocks, 16K-token batches)]
 * LLaMA-style block tail, hidden H, FFN width F, M tokens, bf16, weights [out, in]:
 *   h = O W_o^T + R;  r = rms(h);  [G | U] = r ((h * g) W_gu^T);  a = silu(G) U;  Y = a W_d^T + h
 * (the RMSNorm y = r h g followed by the gate/up GEMM, with r deferred past the GEMM).
 * Two ways to apply the gain g:
 *   - g != NULL (gain broadcast): G1's epilogue also stores u = h * g, the gain broadcast
 *     along each tile as a column vector, and the gate/up GEMM reads u with the
 *     unfolded W_gu.  Needs the u buffer.  No weight preparation.
 *   - g == NULL: W_gu is taken as already folded, W_gu'[n, k] = W_gu[n, k] g[k]
 *     (coda_fold_gain), and the gate/up GEMM reads h. */
typedef struct coda_block_fwd {
  int64_t M, H, F;
  float eps;
  const void* O;        /* [M, H] bf16 */
  const void* R;        /* [M, H] bf16 residual stream input */
  const void* W_o;      /* [H, H] bf16 */
  const void* W_gu;     /* [2F, H] bf16, gate rows first (unfolded if g is set, else folded) */
  const void* W_d;      /* [H, F] bf16 */
  const float* g;       /* optional [H] RMSNorm gain, 16-byte aligned (see above) */
  void* u;              /* [M, H] bf16 out when g is set: h * g, the gate/up GEMM's input */
  void* h;              /* out [M, H] bf16 */
  float* r;             /* out [M] fp32 */
  void* a;              /* out [M, F] bf16 */
  void* Y;              /* out [M, H] bf16 */
  void* Z;              /* optional out [M, 2F] bf16: saved [G | U] (training); NULL = not saved */
  float* Y_partials;    /* optional out [H/256, M] fp32: partial sums of squares of Y; NULL = none */
  float* workspace;     /* [H/256, M] fp32 scratch for the partials of h */
} coda_block_fwd;
CODA_API int coda_block_forward(const coda_block_fwd* io, void* stream);

/* coda_block_forward_noalloc — the same chain for callers that cannot allocate device memory.
 * The pages describe no such call; it exists for deployment, not for the method.
 * Some callers cannot call cudaMalloc at all: a custom operator inside a host runtime that
 * owns the whole device memory pool and hands its operators only their inputs and outputs,
 * or a deployment with a fixed memory budget that forbids allocation after start-up.  Such
 * callers cannot provide the chain's scratch (`workspace`).
 *   - The caller still owns and passes every input and output (O, R, the weights, h, r, a,
 *     Y and the optional Z and Y_partials); `io->workspace` must be NULL.
 *   - The partial sums of squares that G1 writes and the row reduce reads live instead in
 *     a static device array of CODA_NOALLOC_MAX_PARTIALS floats (4 MiB), which every device
 *     that loads the library holds until the process exits.
 *   - Limit: ceil(H / 256) * M <= CODA_NOALLOC_MAX_PARTIALS (M <= 131072 tokens at
 *     H = 2048).  Larger problems, or a non-NULL workspace, return CODA_ERR_SHAPE and
 *     launch nothing.
 *   - Set-up: the first call on each device (in each CUDA context of that device) looks up
 *     the array's device address, with that device current, and caches it.  After a device
 *     reset the next call sees a new context and looks the address up again.
 *   - Sharing: all calls on a device use the same array, which keeps the last call's
 *     contents.  Nothing in it needs clearing (each call writes every partial it reads
 *     before reading it), but calls that overlap on the GPU (unordered streams) race on it.
 *   - It allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 * It issues the same kernels, in the same order, as coda_block_forward with a caller
 * workspace, so its results equal that call's bit for bit. */
#define CODA_NOALLOC_MAX_PARTIALS (1 << 20)
CODA_API int coda_block_forward_noalloc(const coda_block_fwd* io, void* stream);

/* [KuCoin, "El epílogo esconde un tesoro" (the backward inherits the same structure: GEMMs
 * whose epilogues apply the SwiGLU and RMSNorm backward and emit partials)]
 * Backward of coda_block_forward (plain-chain gradients in fused form):
 *   e = r [dA U silu'(G) | dA silu(G)] with dA = dY W_d;  s_i = sum e . Z;  c = r s / H
 *   t = e W_gu;  dh = g t - c h + dY (= dR);  dg = sum_rows h t;  dO = dh W_o
 *   dW_d = dY^T a;  dW_gu[n, k] = g_k (e^T h)[n, k];  dW_o = dh^T O
 * W_gu here is the UNFOLDED gate/up weight (the model parameter itself, not the folded copy
 * the forward reads) and g the RMSNorm gain; dW_gu is the gradient of
 * that unfolded weight.  Weight gradients and dg are fp32; activation gradients bf16. */
typedef struct coda_block_bwd {
  int64_t M, H, F;
  const void* O;       /* [M, H] bf16 */
  const void* W_o;     /* [H, H] bf16 */
  const void* W_gu;    /* [2F, H] bf16, unfolded */
  const void* W_d;     /* [H, F] bf16 */
  const float* g;      /* [H] RMSNorm gain */
  const void* h;       /* saved by the forward: [M, H] bf16 */
  const float* r;      /* [M] */
  const void* Z;       /* [M, 2F] bf16 ([G | U], post-r) */
  const void* a;       /* [M, F] bf16 */
  const void* dY;      /* [M, H] bf16 */
  void* e;             /* out [M, 2F] bf16 */
  void* dh;            /* out [M, H] bf16 (also dR) */
  void* dO;            /* out [M, H] bf16 */
  float* dW_o;         /* out [H, H] */
  float* dW_gu;        /* out [2F, H] */
  float* dW_d;         /* out [H, F] */
  float* dg;           /* out [H] */
  float* c;            /* out [M] */
  float* workspace;    /* coda_workspace_size(CODA_WS_BLOCK_BWD, ...) bytes */
} coda_block_bwd;
CODA_API int coda_block_backward(const coda_block_bwd* io, void* stream);

/* [KuCoin, "El epílogo esconde un tesoro" (r deferred past the GEMM) and "Cinco bloques…"
 * (RoPE as a pairwise transform in the epilogue)]
 * QKV projection with the deferred input-RMSNorm scale and RoPE on Q and K:
 *   QKV = rope(r (h W_qkv'^T)), pos = row mod seq_len, r = rms(h) computed here. */
typedef struct coda_qkv_rope_io {
  int64_t M, H, N;           /* N = (n_q + 2 n_kv) * head_dim */
  int32_t seq_len, head_dim, rope_ncols;   /* rope_ncols = (n_q + n_kv) * head_dim */
  float eps;
  const void* h;             /* [M, H] bf16 */
  const void* W_qkv;         /* [N, H] bf16, gain folded */
  const float* rope_cos; const float* rope_sin;   /* coda_rope_table */
  float* r;                  /* out [M] */
  void* out;                 /* out [M, N] bf16 */
} coda_qkv_rope_io;
CODA_API int coda_qkv_rope(const coda_qkv_rope_io* io, void* stream);

/* [KuCoin, "El epílogo esconde un tesoro" (the backward inherits the structure)]
 * Backward of coda_qkv_rope for an upstream gradient dout of its output (the attention
 * backward's dQ, dK, dV), in fused form:
 *   e = r R(-phi) dout   (rotation transposed on the first rope_ncols columns; coda_rope_backward)
 *   c = r s / H with s = r sum_n dout_n out_n (= sum_n e_n Z_n: rotations keep inner products)
 *   t = e W_qkv;  dh = g t - c h [+ dres];  dg = sum_rows h t;  dW_qkv[n, k] = g_k (e^T h)[n, k]
 * W_qkv is the unfolded weight and g the attention-input RMSNorm gain. */
typedef struct coda_qkv_rope_bwd_io {
  int64_t M, H, N;
  int32_t seq_len, head_dim, rope_ncols;
  const void* h;             /* [M, H] bf16 */
  const float* g;            /* [H] */
  const void* W_qkv;         /* [N, H] bf16, unfolded */
  const float* r;            /* [M] from the forward */
  const void* out;           /* [M, N] bf16 forward output */
  const void* dout;          /* [M, N] bf16 */
  const void* dres;          /* optional [M, H] bf16 gradient arriving on the residual stream */
  const float* rope_cos; const float* rope_sin;
  void* e;                   /* out [M, N] bf16 */
  void* dh;                  /* out [M, H] bf16 */
  float* dW_qkv;             /* out [N, H] fp32 */
  float* dg;                 /* out [H] */
  float* c;                  /* out [M] */
  float* workspace;          /* ceil(M / 32) * H floats */
} coda_qkv_rope_bwd_io;
CODA_API int coda_qkv_rope_backward(const coda_qkv_rope_bwd_io* io, void* stream);

/* [KuCoin, "Cinco bloques…" (RoPE, a pairwise transform; its gradient rotates back)]
 * The row-wise RoPE-backward pass on its own: e = r R(-phi) dout (bf16 [M, N]) and
 * c[i] = r_i^2 sum_n dout_in out_in / H.  The cos/sin tables are those of coda_rope_table,
 * 16-byte aligned (CODA_ERR_ALIGN otherwise); head_dim a multiple of 8. */
CODA_API int coda_rope_backward(const coda_tensor* dout, const coda_tensor* out, const float* r, const float* rope_cos,
                                const float* rope_sin, int32_t seq_len, int32_t head_dim, int32_t rope_ncols,
                                int64_t H, const coda_tensor* e_out, float* c_out, void* stream);

/* [KuCoin, "El «impuesto a la pereza»…" (FP8 makes the matmul faster, so the epilogue work
 * around it weighs more) and "El epílogo esconde un tesoro" (deferred r)]
 * FP8 (e4m3, per-tensor fp32 scales) MLP with deferred r:
 *   Z = r s_x s_w (X_q W_q^T);  a = silu(Z_gate) Z_up;  a_q = e4m3(a / s_a);  amax = max|a|
 *   Y = s_a s_wd (a_q W_dq^T) + h;  Y_partials = partial sums of squares of Y. */
typedef struct coda_mlp_fp8_io {
  int64_t M, H, F;
  float eps, s_x, s_w, s_wd, s_a;
  const void* h;             /* [M, H] bf16: residual input, and source of r */
  const void* X_q;           /* [M, H] e4m3 */
  const void* W_q;           /* [2F, H] e4m3 */
  const void* W_dq;          /* [H, F] e4m3 */
  float* r;                  /* out [M] */
  void* a_q;                 /* out [M, F] e4m3 */
  float* amax;               /* out: 1 float (zeroed by this call on the stream) */
  void* Y;                   /* out [M, H] bf16 */
  float* Y_partials;         /* out [H/256, M] fp32 */
  void* Z;                   /* optional out [M, 2F] bf16: saved [G | U] for the backward; NULL = none */
} coda_mlp_fp8_io;
CODA_API int coda_mlp_fp8(const coda_mlp_fp8_io* io, void* stream);

/* Backward of the FP8 MLP, every GEMM on e4m3 operands with per-tensor scales like the
 * forward's.  The output gradient dY and the SwiGLU-backward output e are quantised with
 * the caller's scales s_dy and s_e (delayed scaling: take them from amax_dy / 448 and
 * amax_e / 448 of an earlier step) [KuCoin, "El epílogo esconde un tesoro" (the backward
 * inherits the epilogue structure); "El «impuesto a la pereza» para entrenar modelos
 * grandes" (FP8 shrinks the GEMM time, so the non-GEMM traffic weighs more)]:
 *   dY_q = e4m3(dY / s_dy);  dA = s_dy s_wd (dY_q W_dq)          (W_dq read MN-major)
 *   e = r [dA U silu'(G) | dA silu(G)];  e_q = e4m3(e / s_e)     (in the dA GEMM's epilogue)
 *   c = r sum_k (s_e e_q) Z / H;  dh = s_e s_w (e_q W_q) - c h + dY
 *   dW_d = s_dy s_a (dY_q^T a_q);  dW = s_e s_x (e_q^T X_q)      (both operands MN-major)
 * dW is the gradient of the effective gate/up weight s_w W_q (the gain, if any, folded in).
 * Six launches: quantise dY, dA GEMM, row reduce, dW_d GEMM, dh GEMM, dW GEMM.  The e4m3
 * quantisations divide by the scale as a multiply by its fp32 reciprocal.  All scales must
 * be > 0 (else CODA_ERR_SHAPE).  M = 0 zeroes dW_d, dW and the two amax outputs; the
 * M-sized pointers may then be NULL. */
typedef struct coda_mlp_fp8_bwd_io {
  int64_t M, H, F;
  float s_x, s_w, s_wd, s_a, s_dy, s_e;
  const void* h;             /* [M, H] bf16 forward input (residual, source of r) */
  const void* X_q;           /* [M, H] e4m3 */
  const void* W_q;           /* [2F, H] e4m3 */
  const void* W_dq;          /* [H, F] e4m3 */
  const void* Z;             /* [M, 2F] bf16 saved by the forward */
  const void* a_q;           /* [M, F] e4m3 saved by the forward */
  const float* r;            /* [M] saved by the forward */
  const void* dY;            /* [M, H] bf16 */
  void* dY_q;                /* out [M, H] e4m3 */
  float* amax_dy;            /* out: max |dY| (zeroed by this call on the stream) */
  void* e_q;                 /* out [M, 2F] e4m3 */
  float* amax_e;             /* out: max |e| before quantisation (zeroed by this call) */
  float* c;                  /* out [M] */
  void* dh;                  /* out [M, H] bf16 */
  float* dW_d;               /* out [H, F] fp32 */
  float* dW;                 /* out [2F, H] fp32 */
  float* workspace;          /* coda_workspace_size(CODA_WS_MLP_FP8_BWD, M, H, F) bytes */
} coda_mlp_fp8_bwd_io;
CODA_API int coda_mlp_fp8_backward(const coda_mlp_fp8_bwd_io* io, void* stream);

/* [KuCoin, "El «impuesto a la pereza»…" (FP8 operands for the matmul)]
 * e4m3 quantisation of a bf16 tensor X (ROW_MAJOR [M, N], N a multiple of 16) into Q
 * (e4m3 ROW_MAJOR [M, N]): Q = e4m3(X * (1 / scale)), round to nearest even, saturating
 * to +-448, 1 / scale taken in fp32; amax (optional) receives the atomic max of |X| (the
 * caller zeroes it).  A bandwidth-bound pass: 3 bytes moved per element. */
CODA_API int coda_quantize_e4m3(const coda_tensor* X, float scale, const coda_tensor* Q, float* amax, void* stream);

/* [KuCoin, "El «impuesto a la pereza»…" (FP4 operands for the matmul; NVFP4 is the 4-bit
 * block-scaled format of these tensor cores)]
 * NVFP4 quantisation of a bf16 tensor X (ROW_MAJOR [R, K], K a multiple of 64) with tensor
 * scale s > 0: for each block of 16 consecutive elements of a row,
 *   sf = e4m3(amax_block / (6 s)),  q = e2m1(x / (sf s))   (q = 0 where sf = 0),
 * both conversions round-to-nearest-even and saturating.  The kernel takes these steps in
 * fp32, as x * (1 / (sf s)) with each product, quotient and reciprocal rounded once, so a
 * value within an fp32 rounding of a rounding midpoint may round the other way than in exact
 * arithmetic.
 * Q (CODA_NVFP4 [R, K]) receives the codes, block_scales the e4m3 scale bytes, amax (optional,
 * zeroed by the caller) the atomic max of |X|.  The SwiGLU epilogue of an NVFP4 GEMM decides
 * its output's codes the same way.
 * Block-scale layout (ceil(R / 128) * (K / 64) * 512 bytes): atoms of 128 rows x 4 blocks;
 * atom (row / 128, kb / 4) starts at byte ((row / 128) * (K / 64) + kb / 4) * 512, and inside
 * it row r, block kb sits at 16 (r % 32) + 4 ((r % 128) / 32) + kb % 4.  So the 16 bytes at
 * 16 i hold rows i, i + 32, i + 64, i + 96 (the order in which the block-scaled MMA reads the
 * scales from TMEM, row m at lane m, column (m % 128) / 32 of a 4-column group): the GEMM's
 * scale warps, one per TMEM lane quarter, fetch their rows' scales with conflict-free loads.
 * Rows from R up to the next multiple of 128 get zero scales. */
CODA_API int coda_quantize_nvfp4(const coda_tensor* X, float s, const coda_tensor* Q, void* block_scales,
                                 float* amax, void* stream);

/* [KuCoin, "El «impuesto a la pereza»…" (FP4 operands) and "El epílogo esconde un tesoro" (the
 * backward inherits the structure: a weight gradient contracts over the tokens)]
 * Transposed NVFP4 quantisation: X (bf16 ROW_MAJOR [R, C]) quantised along its columns into
 * Q = X^T (CODA_NVFP4 [C, R]): for each column c and each block of 16 consecutive rows,
 *   sf = e4m3(amax_block / (6 s)),  Q[c, r] = e2m1(X[r, c] / (sf s)),
 * block scales in the layout described there for the tensor [C, R].  The decisions are taken
 * in fp32 as amax_block * (1 / (6 s)) (the reciprocal rounded once) and X[r, c] times the
 * hardware's approximate reciprocal of sf s (at most one ulp off), so a value within a few
 * fp32 roundings of a rounding midpoint (an exact tie included) may round the other way than
 * in exact arithmetic.  It
 * is the K-major operand of a GEMM that contracts over R, as the block-scaled tensor cores
 * need.  mode CODA_QT_SWIGLU: X is a saved [G | U] ([R, 2C]) and the value quantised is
 * silu(G) U, formed in fp32.  With Q_rows (optional, CODA_NVFP4 [R, C], R a multiple of 128)
 * and its row_block_scales, the same pass also writes the value quantised along its rows (as
 * coda_quantize_nvfp4 would, same s), for a tensor that two GEMMs read along different K.
 * R must be a multiple of 64 and C of 128 (CODA_ERR_SHAPE); amax (optional, zeroed by the
 * caller) receives the atomic max of the quantised values' |x|.  A bandwidth-bound pass: 2 (or
 * 4) bytes read and 9 / 16 (twice that with Q_rows) written per element. */
enum coda_qt_mode { CODA_QT_PLAIN = 0, CODA_QT_SWIGLU = 1 };
CODA_API int coda_quantize_nvfp4_t(const coda_tensor* X, int32_t mode, float s, const coda_tensor* Q,
                                   void* block_scales, const coda_tensor* Q_rows, void* row_block_scales,
                                   float* amax, void* stream);

/* Bytes of the block scales of an NVFP4 tensor [R, K]: ceil(R / 128) * (K / 64) * 512 (the
 * layout at coda_quantize_nvfp4; no counterpart on the pages).  Needs no device. */
CODA_API size_t coda_nvfp4_scale_bytes(int64_t R, int64_t K);

/* [KuCoin, "El «impuesto a la pereza»…" (FP4 makes the matmul faster) and "El epílogo esconde
 * un tesoro" (deferred r; quantisation as an epilogue cast)]
 * NVFP4 MLP with deferred r, the FP8 MLP above with every GEMM operand in NVFP4:
 *   Z = r s_x s_w (X W^T);  a = silu(Z_gate) Z_up;  (a_q, a_sf) = nvfp4(a, s_a);  amax = max|a|
 *   Y = s_a s_wd (a W_d^T) + h;  Y_partials = partial sums of squares of Y
 * X, W, W_d, a are (codes, block scales); s_a is the caller's delayed scale of a (e.g. the
 * previous step's amax / (6 * 448)).  H and F multiples of 256.  Three launches: row RMS,
 * gate/up GEMM + r + SwiGLU + NVFP4 quantisation, down GEMM + residual + partials. */
typedef struct coda_mlp_nvfp4_io {
  int64_t M, H, F;
  float eps, s_x, s_w, s_wd, s_a;
  const void* h;             /* [M, H] bf16: residual input, and source of r */
  const void* X_q;           /* [M, H] NVFP4 codes (M x H / 2 bytes) */
  const void* X_sf;          /* block scales of X */
  const void* W_q;           /* [2F, H] NVFP4 codes, gate rows then up rows (gain folded) */
  const void* W_sf;          /* block scales of W */
  const void* W_dq;          /* [H, F] NVFP4 codes */
  const void* W_dsf;         /* block scales of W_d */
  float* r;                  /* out [M] */
  void* a_q;                 /* out [M, F] NVFP4 codes */
  void* a_sf;                /* out: block scales of a (coda_nvfp4_scale_bytes(M, F)) */
  float* amax;               /* out: 1 float (zeroed by this call on the stream) */
  void* Y;                   /* out [M, H] bf16 */
  float* Y_partials;         /* out [H/256, M] fp32 */
} coda_mlp_nvfp4_io;
CODA_API int coda_mlp_nvfp4(const coda_mlp_nvfp4_io* io, void* stream);

/* [KuCoin, "El epílogo esconde un tesoro" (the backward inherits the structure) and "El
 * «impuesto a la pereza»…" (FP4 operands for the matmul)]
 * Backward of the NVFP4 MLP for an output gradient dY, every GEMM on NVFP4 operands.  The
 * block-scaled tensor cores take both operands blocked along the GEMM's K, so each operand is
 * quantised along the K of the GEMM that reads it:
 *   dY_r = nvfp4 of dY along its rows, dY_c along its columns (tensor scale s_dy)
 *   dA = s_dy s_wdt (dY_r W_dT^T);  e = r [dA U silu'(G) | dA silu(G)] (bf16, from the saved Z)
 *   s_i = sum_k e_ik Z_ik;  c = r s / H
 *   e_r, e_c = e along its rows / columns (s_e);  a_c = silu(G) U along its columns (s_a);
 *   x_c = h along its columns (s_x)
 *   dh = s_e s_wt (e_r W_guT^T) - c h + dY
 *   dW_d = s_dy s_a (dY_c a_c^T)  [H, F];  dW = s_e s_x (e_c x_c^T)  [2F, H]   (fp32)
 * W_guT ([H, 2F]) and W_dT ([F, H]) are the gate/up and down weights quantised transposed,
 * along 2F and H (coda_quantize_nvfp4_t of W_gu and W_d; once per weight update), with tensor
 * scales s_wt and s_wdt.  s_dy and s_e are the caller's delayed scales (e.g. amax_dy / 2688
 * and amax_e / 2688 of an earlier step), s_a the forward's, s_x that of h.  The caller owns
 * every intermediate; the NVFP4 ones are (codes, block scales) pairs of the sizes given by
 * their shapes (coda_nvfp4_scale_bytes).  M must be a multiple of 256 (the weight gradients
 * contract over the tokens), H and F multiples of 256: CODA_ERR_SHAPE otherwise.  Nine
 * launches: dY quantised both ways in one pass, the dA GEMM with the SwiGLU-backward epilogue,
 * the row reduce, e quantised both ways in one pass, silu(G) U and h along their columns, the
 * dW_d, dh and dW GEMMs. */
typedef struct coda_mlp_nvfp4_bwd_io {
  int64_t M, H, F;
  float s_x, s_wt, s_wdt, s_a, s_dy, s_e;
  const void* h;             /* [M, H] bf16 */
  const void* W_guT;         /* NVFP4 [H, 2F] codes */
  const void* W_guT_sf;      /* its block scales */
  const void* W_dT;          /* NVFP4 [F, H] codes */
  const void* W_dT_sf;
  const void* Z;             /* [M, 2F] bf16: saved [G | U] */
  const float* r;            /* [M] */
  const void* dY;            /* [M, H] bf16 */
  void* dY_r;                /* out NVFP4 [M, H] codes, and scales */
  void* dY_r_sf;
  void* dY_c;                /* out NVFP4 [H, M] */
  void* dY_c_sf;
  void* e;                   /* out [M, 2F] bf16 */
  void* e_r;                 /* out NVFP4 [M, 2F] */
  void* e_r_sf;
  void* e_c;                 /* out NVFP4 [2F, M] */
  void* e_c_sf;
  void* a_c;                 /* out NVFP4 [F, M] */
  void* a_c_sf;
  void* x_c;                 /* out NVFP4 [H, M] */
  void* x_c_sf;
  float* amax_dy;            /* out: max |dY| (zeroed by this call on the stream) */
  float* amax_e;             /* out: max |e| (likewise) */
  float* c;                  /* out [M] */
  void* dh;                  /* out [M, H] bf16 */
  float* dW_d;               /* out [H, F] fp32 */
  float* dW;                 /* out [2F, H] fp32 */
  float* workspace;          /* coda_workspace_size(CODA_WS_MLP_NVFP4_BWD, M, H, F) bytes */
} coda_mlp_nvfp4_bwd_io;
CODA_API int coda_mlp_nvfp4_backward(const coda_mlp_nvfp4_bwd_io* io, void* stream);

/* ------------------------------------------------------------ LM head + cross-entropy
 * Final RMSNorm, LM head and mean cross-entropy, with the logits never stored
 * [KuCoin, "El epílogo esconde un tesoro" (cross-entropy rewritten as an epilogue),
 * "Cinco bloques…" (block log-sum-exp, max / sum-exp state), "hoja de referencia"]:
 *   u = h * g, r = rms(h)                        (coda_rms_gain)
 *   z = r (u W_v^T): per tile online (max, sum-exp) and the target logit   (XENT GEMM)
 *   lse, loss_i = lse_i - z[i, target_i], mean  (coda_xent_combine) */
typedef struct coda_lm_head_xent_io {
  int64_t M, H, V;
  float eps;
  const void* h;            /* [M, H] bf16 final hidden state */
  const float* g;           /* [H] final RMSNorm gain, 16-byte aligned */
  const void* W_v;          /* [V, H] bf16 LM-head weight */
  const int32_t* targets;   /* [M] target classes in [0, V) */
  void* u;                  /* out [M, H] bf16 = h * g */
  float* r;                 /* out [M] */
  float* lse;               /* out [M] */
  float* loss;              /* out [M] per-row loss */
  float* loss_mean;         /* out [1] */
  float* workspace;         /* coda_workspace_size(CODA_WS_XENT_FWD, M, H, V) bytes */
} coda_lm_head_xent_io;
CODA_API int coda_lm_head_xent_forward(const coda_lm_head_xent_io* io, void* stream);

/* Backward for an upstream gradient dloss of the mean loss (fused forms):
 *   e = r dloss (exp(z - lse) - onehot(target)) / M   (logits recomputed in the epilogue)
 *   s_i = sum_v e_iv z_iv, c = r s / H;  t = e W_v;  dh = g t - c h;  dg = sum_rows h t
 *   dW_v = e^T u */
typedef struct coda_lm_head_xent_bwd_io {
  int64_t M, H, V;
  float dloss;
  const void* h;            /* [M, H] bf16 */
  const float* g;           /* [H] */
  const void* W_v;          /* [V, H] bf16 */
  const int32_t* targets;   /* [M] */
  const void* u;            /* saved by the forward: [M, H] bf16 */
  const float* r;           /* saved: [M] */
  const float* lse;         /* saved: [M] */
  void* e;                  /* out [M, V] bf16 */
  void* dh;                 /* out [M, H] bf16 */
  float* dW_v;              /* out [V, H] fp32 */
  float* dg;                /* out [H] */
  float* c;                 /* out [M] */
  float* workspace;         /* coda_workspace_size(CODA_WS_XENT_BWD, M, H, V) bytes */
} coda_lm_head_xent_bwd_io;
CODA_API int coda_lm_head_xent_backward(const coda_lm_head_xent_bwd_io* io, void* stream);

/* Bytes of fp32 scratch a chain needs (caller allocates): the partial buffers of the
 * partial + light-reduce pattern [KuCoin, "El epílogo esconde un tesoro"].  The third size
 * is F for the block chains and V for the cross-entropy chains.  Returns 0 for an unknown
 * `which` or negative sizes.  Allocates nothing and needs no device. */
enum coda_workspace_kind {
  CODA_WS_BLOCK_FWD = 0,
  CODA_WS_BLOCK_BWD = 1,
  CODA_WS_XENT_FWD = 2,
  CODA_WS_XENT_BWD = 3,
  CODA_WS_MLP_FP8_BWD = 4,
  CODA_WS_MLP_NVFP4_BWD = 5
};
CODA_API size_t coda_workspace_size(int32_t which, int64_t M, int64_t H, int64_t F);

/* ------------------------------------------------------------------ device status
 * The pages describe no failure detection; this is the library's own: every kernel wait is
 * bounded in time and a wait that runs out records where, instead of hanging.
 * Synchronises `stream`, then reads and clears the current device's status word.
 * *site receives 0 or the site code of the first kernel wait that ran out of time
 * (1 producer / empty stage, 2 MMA / free accumulator, 3 MMA / full stage,
 * 4 epilogue / accumulator, 5 epilogue / side input, 6 NVFP4 scale warp / block scales in
 * shared memory, 7 MMA / NVFP4 block scales in TMEM).  Returns CODA_OK,
 * CODA_ERR_DEVICE_TIMEOUT, or CODA_ERR_LAUNCH if the stream itself reports an error. */
CODA_API int coda_get_device_status(void* stream, int32_t* site);

/* Per-wait time limit of every kernel wait (default 2000 ms, or CODA_WATCHDOG_MS); the
 * library's own failure detection (no counterpart on the pages).  0 returns CODA_ERR_SHAPE. */
CODA_API int coda_set_watchdog_ms(uint32_t ms);

/* No counterpart on the pages (a launch property of this library).
 * Launch overlap (default on; CODA_LAUNCH_OVERLAP=0 in the environment turns it off): every
 * kernel of the library is launched with a programmatic dependency on the previous kernel of
 * the stream, signals at entry and waits for that kernel's completion before its first global
 * memory access, so stream order is kept while the launch itself overlaps the previous kernel's
 * tail.  enable = 0 gives plain stream serialisation.  Other values: CODA_ERR_SHAPE. */
CODA_API int coda_set_launch_overlap(int32_t enable);

/* No counterpart on the pages (tests the library's own failure detection).
 * Test hook for the watchdog: the next coda_gemm_epilogue call drops its first k-block, so
 * the MMA wait runs out of time and the kernel returns through the abort path.  Cleared after
 * one call.  enable: 0 off; 1 every producer drops it; for the CTA-pair GEMMs (every bf16,
 * e4m3 and NVFP4 program) 2 only the second CTA of each pair drops it (the leader has armed
 * that phase for bytes that never come) and 3 only the leader does (the second CTA's bytes
 * land on a phase nobody armed).  Other values: CODA_ERR_SHAPE. */
CODA_API int coda_inject_dropped_stage(int32_t enable);

/* No counterpart on the pages (utilities).  Number of SMs of the current device
 * (CODA_ERR_NO_DEVICE without an sm_103 device), the message of a status code, and the
 * library's build tag. */
CODA_API int coda_device_sm_count(int32_t* sms);
CODA_API const char* coda_status_string(int status);
CODA_API const char* coda_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CODA_H_ */
