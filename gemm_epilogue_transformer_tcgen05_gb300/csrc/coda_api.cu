// C ABI of the GEMM-epilogue library: argument checks, epilogue-program matching, TMA
// descriptor encoding, launches, and the block chains built from those launches.
// The operations follow "CODA: new research optimizes Transformer training with
// GEMM-epilogue programming" (kucoin.com news flash), sections "El epílogo esconde un
// tesoro" (deferred r, partial RMS, backward) and "Cinco bloques y un lenguaje LEGO"
// (primitive kinds); see include/coda.h for each call's contract.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/coda.h"
#include "coda_internal.h"

using namespace coda;

namespace {

// Device status word read by coda_get_device_status.  One per device (module global);
// its address is looked up once per device and passed to every kernel.
__device__ int g_device_status;

struct DevState {
  bool init;
  bool ok;
  int sms;
  int* status;
};
constexpr int kMaxDevices = 64;
DevState g_dev[kMaxDevices];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::atomic<uint32_t> g_watchdog_ms{0};
std::atomic<int> g_inject_once{0};

int ensure_device(DevState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return CODA_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  DevState& d = g_dev[dev];
  if (!d.init) {
    d.init = true;
    d.ok = false;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return CODA_ERR_NO_DEVICE;
    }
    if (major != 10 || minor != 3) return CODA_ERR_NO_DEVICE;
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr) {
        cudaGetLastError();
        return CODA_ERR_NO_DEVICE;
      }
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess || addr == nullptr) {
      cudaGetLastError();
      return CODA_ERR_NO_DEVICE;
    }
    d.status = static_cast<int*>(addr);
    d.sms = sms;
    if (g_watchdog_ms == 0) {
      const char* env = std::getenv("CODA_WATCHDOG_MS");
      long v = env ? std::strtol(env, nullptr, 10) : 0;
      g_watchdog_ms = v > 0 ? (uint32_t)v : 2000u;
    }
    d.ok = true;
  }
  if (!d.ok) return CODA_ERR_NO_DEVICE;
  *out = &d;
  return CODA_OK;
}

// element bytes (NVFP4: 1, the byte holding two codes; sizes in bytes are halved where used)
int esize(int dt) { return dt == CODA_F32 ? 4 : dt == CODA_BF16 ? 2 : (dt == CODA_E4M3 || dt == CODA_NVFP4) ? 1 : 0; }
int to_dt(int dt) { return dt == CODA_F32 ? DT_F32 : dt == CODA_BF16 ? DT_BF16 : dt == CODA_NVFP4 ? DT_E2M1 : DT_E4M3; }
// bytes of n elements along a row
int64_t row_bytes(int dt, int64_t n) { return dt == CODA_NVFP4 ? n / 2 : n * esize(dt); }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
const int64_t kMaxDim = (int64_t(1) << 31) - 1;

// Checks a tensor's pointer, dtype, alignment and leading dimension.
// An empty tensor (rows or cols = 0) may have a NULL pointer.
int check_tensor(const coda_tensor* t, bool allow_col) {
  if (!t) return CODA_ERR_NULL;
  if (esize(t->dtype) == 0) return CODA_ERR_DTYPE;
  if (t->layout != CODA_ROW_MAJOR && !(allow_col && t->layout == CODA_COL_MAJOR)) return CODA_ERR_SHAPE;
  if (t->rows < 0 || t->cols < 0 || t->rows > kMaxDim || t->cols > kMaxDim) return CODA_ERR_SHAPE;
  if (t->rows == 0 || t->cols == 0) return CODA_OK;
  if (!t->ptr) return CODA_ERR_NULL;
  const int64_t inner = t->layout == CODA_ROW_MAJOR ? t->cols : t->rows;
  if (t->ld < inner || t->ld < 1) return CODA_ERR_SHAPE;
  if (t->dtype == CODA_NVFP4 && (t->layout != CODA_ROW_MAJOR || t->cols % 2 != 0 || t->ld % 2 != 0))
    return CODA_ERR_SHAPE;
  if (!aligned16(t->ptr) || row_bytes(t->dtype, t->ld) % 16 != 0) return CODA_ERR_ALIGN;
  return CODA_OK;
}

// 2-D tiled tensor map over storage [outer][ld] with `inner` valid elements per row.
int encode_2d(CUtensorMap* m, int dtype, const void* ptr, int64_t inner, int64_t outer, int64_t ld, uint32_t box_in,
              uint32_t box_out) {
  CUtensorMapDataType t = dtype == CODA_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                          : dtype == CODA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                               : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const uint32_t row_bytes = box_in * (uint32_t)esize(dtype);
  CUtensorMapSwizzle sw = row_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                          : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                          : row_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                            : CU_TENSOR_MAP_SWIZZLE_NONE;
  cuuint64_t dims[2] = {(cuuint64_t)(inner > 0 ? inner : 1), (cuuint64_t)(outer > 0 ? outer : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * esize(dtype))};
  cuuint32_t box[2] = {box_in, box_out};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, t, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CODA_OK : CODA_ERR_LAUNCH;
}

// 3-D map of a ROW_MAJOR [rows, 2 * half] tensor whose two column halves (gate, up) are copied
// together: dims {half, rows, 2} (strides: a row, then a half), box {box_in, 32, 2}, i.e. the
// two 32-row blocks of the halves one after the other, each swizzled like a 2-D box.
int encode_pair(CUtensorMap* m, int dtype, const void* ptr, int64_t half, int64_t rows, int64_t ld,
                uint32_t box_in = 32) {
  const int es = esize(dtype);
  const uint32_t row_bytes = box_in * (uint32_t)es;
  CUtensorMapSwizzle sw = row_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                          : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                            : CU_TENSOR_MAP_SWIZZLE_32B;
  CUtensorMapDataType t = dtype == CODA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  cuuint64_t dims[3] = {(cuuint64_t)(half > 0 ? half : 1), (cuuint64_t)(rows > 0 ? rows : 1), 2};
  cuuint64_t strides[2] = {(cuuint64_t)(ld * es), (cuuint64_t)(half * es)};
  cuuint32_t box[3] = {box_in, 32, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, t, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CODA_OK : CODA_ERR_LAUNCH;
}

// Map over NVFP4 block-scale atoms: n_atoms rows of 512 bytes (128 uint32), box of 4 atoms.
int encode_atoms(CUtensorMap* m, const void* ptr, int64_t n_atoms) {
  cuuint64_t dims[2] = {128, (cuuint64_t)(n_atoms > 0 ? n_atoms : 1)};
  cuuint64_t strides[1] = {512};
  cuuint32_t box[2] = {128, 4};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CODA_OK : CODA_ERR_LAUNCH;
}

// ------------------------------------------------------------- program matching
struct Item {
  int op;
  bool optional;
};
struct ProgramTemplate {
  int epi;
  int n;
  Item items[6];
};
const ProgramTemplate kPrograms[] = {
    {EPI_STORE, 2, {{CODA_OP_TENSOR_SCALE, true}, {CODA_OP_COL_SCALE, true}}},
    {EPI_RESID,
     4,
     {{CODA_OP_TENSOR_SCALE, true},
      {CODA_OP_ADD_SIDE, false},
      {CODA_OP_ROW_SUMSQ_PARTIAL, true},
      {CODA_OP_STORE_COL_SCALED, true}}},
    {EPI_ROWSCALE, 2, {{CODA_OP_TENSOR_SCALE, true}, {CODA_OP_ROW_SCALE, false}}},
    {EPI_SWIGLU,
     5,
     {{CODA_OP_TENSOR_SCALE, true},
      {CODA_OP_ROW_SCALE, true},
      {CODA_OP_STORE_AUX, true},
      {CODA_OP_SWIGLU, false},
      {CODA_OP_AMAX, true}}},
    {EPI_ROPE, 3, {{CODA_OP_TENSOR_SCALE, true}, {CODA_OP_ROW_SCALE, true}, {CODA_OP_ROPE, false}}},
    {EPI_SWIGLU_BWD,
     5,
     {{CODA_OP_TENSOR_SCALE, true},
      {CODA_OP_SWIGLU_BWD, false},
      {CODA_OP_ROW_SCALE, true},
      {CODA_OP_ROW_DOT_PARTIAL, false},
      {CODA_OP_AMAX, true}}},
    {EPI_RMSBWD,
     3,
     {{CODA_OP_TENSOR_SCALE, true}, {CODA_OP_RMSBWD_COMBINE, false}, {CODA_OP_COL_DOT_PARTIAL, true}}},
    {EPI_XENT, 3, {{CODA_OP_TENSOR_SCALE, true}, {CODA_OP_ROW_SCALE, true}, {CODA_OP_XENT_PARTIAL, false}}},
    {EPI_XENT_BWD,
     4,
     {{CODA_OP_TENSOR_SCALE, true},
      {CODA_OP_ROW_SCALE, true},
      {CODA_OP_XENT_BWD, false},
      {CODA_OP_ROW_DOT_PARTIAL, false}}},
};

// Returns the compiled program index and the set of ops present (bit op), or -1.
int match_program(const coda_epilogue_program* prog, uint32_t* present) {
  const int n = prog ? prog->n_ops : 0;
  if (n < 0 || n > CODA_MAX_OPS) return -1;
  for (const ProgramTemplate& t : kPrograms) {
    int pos = 0;
    uint32_t seen = 0;
    bool ok = true;
    for (int i = 0; i < t.n && ok; ++i) {
      if (pos < n && prog->ops[pos] == t.items[i].op) {
        seen |= 1u << t.items[i].op;
        ++pos;
      } else if (!t.items[i].optional) {
        ok = false;
      }
    }
    if (ok && pos == n) {
      *present = seen;
      return t.epi;
    }
  }
  return -1;
}

}  // namespace

namespace coda {
std::atomic<int> g_launch_overlap = [] {
  const char* e = std::getenv("CODA_LAUNCH_OVERLAP");
  return (e && e[0] == '0') ? 0 : 1;
}();

const VariantEntry* find_variant(const VariantKey& k) {
  const VariantEntry* tables[5] = {g_variants_fwd, g_variants_bwd, g_variants_lowp, g_variants_fp8, g_variants_fp4};
  const int counts[5] = {g_num_variants_fwd, g_num_variants_bwd, g_num_variants_lowp, g_num_variants_fp8,
                         g_num_variants_fp4};
  for (int t = 0; t < 5; ++t)
    for (int i = 0; i < counts[t]; ++i) {
      const VariantKey& v = tables[t][i].key;
      if (v.kind == k.kind && v.epi == k.epi && v.a_mn == k.a_mn && v.b_mn == k.b_mn && v.out_dt == k.out_dt &&
          v.side_dt == k.side_dt && v.aux == k.aux)
        return &tables[t][i];
    }
  return nullptr;
}
}  // namespace coda

// =====================================================================================
extern "C" {

const char* coda_version(void) { return "coda-gb300 sm_103a 1"; }

const char* coda_status_string(int s) {
  switch (s) {
    case CODA_OK: return "ok";
    case CODA_ERR_NULL: return "a required pointer is NULL";
    case CODA_ERR_SHAPE: return "inconsistent or unsupported sizes";
    case CODA_ERR_ALIGN: return "base address or leading dimension not 16-byte aligned";
    case CODA_ERR_DTYPE: return "unsupported dtype combination";
    case CODA_ERR_UNSUPPORTED_PROGRAM: return "epilogue program has no compiled variant";
    case CODA_ERR_LAUNCH: return "CUDA launch or TMA descriptor encoding failed";
    case CODA_ERR_DEVICE_TIMEOUT: return "a kernel wait ran out of time";
    case CODA_ERR_NO_DEVICE: return "no sm_103 device current (or driver entry point missing)";
    default: return "unknown status";
  }
}

int coda_set_launch_overlap(int32_t enable) {
  if (enable != 0 && enable != 1) return CODA_ERR_SHAPE;
  coda::g_launch_overlap = enable;
  return CODA_OK;
}

int coda_set_watchdog_ms(uint32_t ms) {
  if (ms == 0) return CODA_ERR_SHAPE;
  g_watchdog_ms = ms;
  return CODA_OK;
}

int coda_inject_dropped_stage(int32_t enable) {
  if (enable < 0 || enable > 3) return CODA_ERR_SHAPE;
  g_inject_once = enable;
  return CODA_OK;
}

int coda_device_sm_count(int32_t* sms) {
  if (!sms) return CODA_ERR_NULL;
  DevState* d;
  int st = ensure_device(&d);
  if (st != CODA_OK) return st;
  *sms = d->sms;
  return CODA_OK;
}

int coda_get_device_status(void* stream, int32_t* site) {
  if (!site) return CODA_ERR_NULL;
  DevState* d;
  int st = ensure_device(&d);
  if (st != CODA_OK) return st;
  *site = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  int v = 0;
  if (cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return CODA_ERR_LAUNCH;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(d->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return CODA_ERR_LAUNCH;
    *site = v;
    return CODA_ERR_DEVICE_TIMEOUT;
  }
  return CODA_OK;
}

// ab_ready: the caller guarantees that the kernel issued just before this one on the stream
// writes neither A nor W (the chains know this; the public entry point does not).
static int gemm_epilogue_impl(const coda_tensor* A, const coda_tensor* W, const coda_epilogue_program* prog,
                              const coda_side_inputs* side, const coda_tensor* out, const coda_aux_outputs* aux,
                              void* stream, bool ab_ready) {
  int st;
  if ((st = check_tensor(A, true)) != CODA_OK) return st;
  if ((st = check_tensor(W, true)) != CODA_OK) return st;
  uint32_t present = 0;
  const int epi = match_program(prog, &present);
  if (epi < 0) return CODA_ERR_UNSUPPORTED_PROGRAM;
  if (epi == EPI_XENT) {   // the logits are never stored: out only gives their shape
    if (!out) return CODA_ERR_NULL;
    if (out->rows < 0 || out->cols < 0 || out->rows > kMaxDim || out->cols > kMaxDim) return CODA_ERR_SHAPE;
  } else if ((st = check_tensor(out, false)) != CODA_OK) {
    return st;
  }
  auto has = [&](int op) { return (present >> op) & 1u; };

  // operand kind
  if (A->dtype != W->dtype) return CODA_ERR_DTYPE;
  const int kind = A->dtype == CODA_BF16   ? KIND_BF16
                   : A->dtype == CODA_F32  ? KIND_TF32
                   : A->dtype == CODA_NVFP4 ? KIND_NVFP4
                                            : KIND_E4M3;
  const bool fp4 = kind == KIND_NVFP4;
  const bool a_mn = A->layout == CODA_COL_MAJOR, b_mn = W->layout == CODA_COL_MAJOR;

  const int64_t M = A->rows, K = A->cols;
  if (W->cols != K) return CODA_ERR_SHAPE;
  int64_t N;
  if (epi == EPI_SWIGLU) {
    N = out->cols;
    if (W->rows != 2 * N || N % 128 != 0) return CODA_ERR_SHAPE;
  } else if (epi == EPI_SWIGLU_BWD) {
    N = W->rows;
    if (out->cols != 2 * N) return CODA_ERR_SHAPE;
  } else {
    N = W->rows;
    if (out->cols != N) return CODA_ERR_SHAPE;
  }
  if (out->rows != M) return CODA_ERR_SHAPE;
  if (N % 32 != 0) return CODA_ERR_SHAPE;
  if (M == 0 || N == 0) return CODA_OK;
  if (K < 1) return CODA_ERR_SHAPE;
  if (fp4 && K % 256 != 0) return CODA_ERR_SHAPE;

  // side inputs and aux outputs the program needs
  const coda_side_inputs zero_side{};
  const coda_aux_outputs zero_aux{};
  const coda_side_inputs& sd = side ? *side : zero_side;
  const coda_aux_outputs& ax = aux ? *aux : zero_aux;
  int side_dt = kind == KIND_TF32 ? DT_F32 : DT_BF16;
  if (epi == EPI_RESID) {
    if ((st = check_tensor(sd.residual, false)) != CODA_OK) return st;
    if (sd.residual->rows != M || sd.residual->cols != N) return CODA_ERR_SHAPE;
    side_dt = to_dt(sd.residual->dtype);
  }
  if (epi == EPI_SWIGLU_BWD) {
    if ((st = check_tensor(sd.aux_in, false)) != CODA_OK) return st;
    if (sd.aux_in->rows != M || sd.aux_in->cols != 2 * N) return CODA_ERR_SHAPE;
    side_dt = to_dt(sd.aux_in->dtype);
  }
  if (epi == EPI_RMSBWD) {
    if ((st = check_tensor(sd.aux_in, false)) != CODA_OK) return st;
    if (sd.aux_in2 && (st = check_tensor(sd.aux_in2, false)) != CODA_OK) return st;
    if (sd.aux_in->rows != M || sd.aux_in->cols != N) return CODA_ERR_SHAPE;
    if (sd.aux_in2) {
      if (sd.aux_in2->rows != M || sd.aux_in2->cols != N) return CODA_ERR_SHAPE;
      if (sd.aux_in->dtype != sd.aux_in2->dtype) return CODA_ERR_DTYPE;
    }
    side_dt = to_dt(sd.aux_in->dtype);
    if (!sd.row_coef) return CODA_ERR_NULL;
    if (sd.col_scale && !aligned16(sd.col_scale)) return CODA_ERR_ALIGN;
    if (has(CODA_OP_COL_DOT_PARTIAL) && !sd.col_scale) return CODA_ERR_NULL;   // dg needs the gain
  }
  if (has(CODA_OP_ROW_SCALE) && !sd.row_scale) return CODA_ERR_NULL;
  if (has(CODA_OP_COL_SCALE) || has(CODA_OP_STORE_COL_SCALED)) {
    if (!sd.col_scale) return CODA_ERR_NULL;
    if (!aligned16(sd.col_scale)) return CODA_ERR_ALIGN;
  }
  const bool want_aux = has(CODA_OP_STORE_AUX) || has(CODA_OP_STORE_COL_SCALED);
  if (want_aux) {
    if ((st = check_tensor(ax.store_aux, false)) != CODA_OK) return st;
    const int64_t aux_cols = epi == EPI_SWIGLU ? 2 * N : N;
    if (ax.store_aux->rows != M || ax.store_aux->cols != aux_cols || ax.store_aux->dtype != CODA_BF16)
      return CODA_ERR_SHAPE;
  }
  if (has(CODA_OP_AMAX) && !ax.amax) return CODA_ERR_NULL;
  if (epi == EPI_XENT || epi == EPI_XENT_BWD) {
    if (!sd.row_index) return CODA_ERR_NULL;
    if (epi == EPI_XENT && (!ax.row_partials || !ax.row_partials2 || !ax.row_values)) return CODA_ERR_NULL;
    if (epi == EPI_XENT && ax.row_partials_ld < M) return CODA_ERR_SHAPE;
    if (epi == EPI_XENT_BWD && !sd.row_coef) return CODA_ERR_NULL;
  }
  if (has(CODA_OP_ROW_SUMSQ_PARTIAL) || has(CODA_OP_ROW_DOT_PARTIAL)) {
    if (!ax.row_partials) return CODA_ERR_NULL;
    if (ax.row_partials_ld < M) return CODA_ERR_SHAPE;
  }
  if (has(CODA_OP_COL_DOT_PARTIAL)) {
    if (!ax.col_partials) return CODA_ERR_NULL;
    if (ax.col_partials_ld < N) return CODA_ERR_SHAPE;   // rows: one per 32-row slab, ceil(M / 32)
  }
  if (has(CODA_OP_ROPE)) {
    const int hd = sd.rope_head_dim;
    if (!(hd == 32 || hd == 64 || hd == 128 || hd == 256)) return CODA_ERR_SHAPE;
    if (sd.rope_ncols < 0 || sd.rope_ncols % hd != 0 || sd.rope_ncols > N || sd.rope_seq_len < 1)
      return CODA_ERR_SHAPE;
    if (!sd.rope_cos || !sd.rope_sin) return CODA_ERR_NULL;
    if (!aligned16(sd.rope_cos) || !aligned16(sd.rope_sin)) return CODA_ERR_ALIGN;
  }
  if (out->dtype == CODA_E4M3 && epi != EPI_SWIGLU && epi != EPI_SWIGLU_BWD) return CODA_ERR_DTYPE;
  if (out->dtype == CODA_NVFP4) {   // the NVFP4 SwiGLU output: codes, block scales, tensor scale
    if (!fp4 || epi != EPI_SWIGLU) return CODA_ERR_DTYPE;
    if (!ax.out_block_scales) return CODA_ERR_NULL;
    if (!aligned16(ax.out_block_scales)) return CODA_ERR_ALIGN;
    if (!(sd.out_fp4_scale > 0.f) || !(sd.out_fp4_scale < INFINITY)) return CODA_ERR_SHAPE;
  }
  if (fp4) {
    if (!sd.a_block_scales || !sd.w_block_scales) return CODA_ERR_NULL;
    if (!aligned16(sd.a_block_scales) || !aligned16(sd.w_block_scales)) return CODA_ERR_ALIGN;
  }
  if (epi == EPI_SWIGLU_BWD && has(CODA_OP_AMAX) && out->dtype != CODA_E4M3) return CODA_ERR_UNSUPPORTED_PROGRAM;
  if (out->dtype == CODA_E4M3 && !(sd.out_scale > 0.f)) return CODA_ERR_SHAPE;   // 1 / scale of the codes

  const VariantKey key{kind, epi, a_mn ? 1 : 0, b_mn ? 1 : 0, to_dt(out->dtype), side_dt, want_aux ? 1 : 0};
  const VariantEntry* var = find_variant(key);
  if (!var) return CODA_ERR_DTYPE;
  const int64_t tile_rows = (int64_t)BM * var->cg;
  const int64_t m_tiles = (M + tile_rows - 1) / tile_rows;
  const int64_t n_tiles = (N + var->bn_out - 1) / var->bn_out;

  DevState* d;
  if ((st = ensure_device(&d)) != CODA_OK) return st;

  GemmLaunch L;
  std::memset(&L, 0, sizeof(L));
  const int op_bytes = esize(A->dtype);
  const uint32_t bk = (uint32_t)(128 / op_bytes);
  // A: K-major box {bk, 128}; MN-major (stored [K][M]) box {128 bytes of M, bk}.  NVFP4
  // operands are mapped as bytes (two codes each): box {128 bytes, rows}.
  const uint32_t mn_atom = (uint32_t)(128 / op_bytes);
  if (fp4)
    st = encode_2d(&L.tmA, CODA_E4M3, A->ptr, K / 2, M, A->ld / 2, 128, 128);
  else if (a_mn)
    st = encode_2d(&L.tmA, A->dtype, A->ptr, M, K, A->ld, mn_atom, (uint32_t)var->bk);   // one stage's K rows
  else
    st = encode_2d(&L.tmA, A->dtype, A->ptr, K, M, A->ld, bk, 128);
  if (st != CODA_OK) return st;
  if (fp4)
    st = encode_2d(&L.tmB, CODA_E4M3, W->ptr, K / 2, W->rows, W->ld / 2, 128, (uint32_t)var->b_box);
  else if (b_mn)
    st = encode_2d(&L.tmB, W->dtype, W->ptr, W->rows, K, W->ld, mn_atom, (uint32_t)var->bk);
  else
    st = encode_2d(&L.tmB, W->dtype, W->ptr, K, W->rows, W->ld, bk, (uint32_t)var->b_box);
  if (st != CODA_OK) return st;
  if (fp4) {
    // block scales: rows of 512-byte atoms (as 128 uint32), 4 atoms (one stage) per copy
    const int64_t kc = K / 64;
    if ((st = encode_atoms(&L.tmSFA, sd.a_block_scales, (M + 127) / 128 * kc)) != CODA_OK) return st;
    if ((st = encode_atoms(&L.tmSFB, sd.w_block_scales, (W->rows + 127) / 128 * kc)) != CODA_OK) return st;
  }
  if (out->dtype == CODA_NVFP4) {
    if ((st = encode_2d(&L.tmOut, CODA_E4M3, out->ptr, N / 2, M, out->ld / 2, 16, 32)) != CODA_OK) return st;
  } else if (epi == EPI_SWIGLU_BWD) {   // e: both halves, ow chunks of 32 columns per store
    if ((st = encode_pair(&L.tmOut, out->dtype, out->ptr, N, M, out->ld, 32u * var->ow)) != CODA_OK) return st;
  } else if (epi != EPI_XENT && (st = encode_2d(&L.tmOut, out->dtype, out->ptr, out->cols, M, out->ld,
                                                32u * var->ow, 32)) != CODA_OK) {
    return st;
  }
  if (epi == EPI_RESID) {
    const coda_tensor* r = sd.residual;
    if ((st = encode_2d(&L.tmSide0, r->dtype, r->ptr, r->cols, M, r->ld, 32, 32)) != CODA_OK) return st;
  } else if (epi == EPI_SWIGLU_BWD) {
    const coda_tensor* z = sd.aux_in;   // Z = [G | U]: both halves of a chunk in one copy
    if ((st = encode_pair(&L.tmSide0, z->dtype, z->ptr, N, M, z->ld)) != CODA_OK) return st;
  } else if (epi == EPI_SWIGLU_BWD || epi == EPI_RMSBWD) {
    const coda_tensor* r = sd.aux_in;
    if ((st = encode_2d(&L.tmSide0, r->dtype, r->ptr, r->cols, M, r->ld, 32, 32)) != CODA_OK) return st;
    if (epi == EPI_RMSBWD && sd.aux_in2) {
      const coda_tensor* r2 = sd.aux_in2;
      if ((st = encode_2d(&L.tmSide1, r2->dtype, r2->ptr, r2->cols, M, r2->ld, 32, 32)) != CODA_OK) return st;
    }
  }
  if (want_aux && epi == EPI_SWIGLU) {
    const coda_tensor* z = ax.store_aux;   // saved Z = [G | U]: both halves of a store group in one copy
    if ((st = encode_pair(&L.tmAux, z->dtype, z->ptr, N, M, z->ld, 32u * var->ow)) != CODA_OK) return st;
  } else if (want_aux) {
    const coda_tensor* z = ax.store_aux;
    if ((st = encode_2d(&L.tmAux, z->dtype, z->ptr, z->cols, M, z->ld, 32u * var->ow, 32)) != CODA_OK) return st;
  }

  GemmParams& p = L.p;
  p.M = (int)M;
  p.N = (int)N;
  p.K = (int)K;
  p.m_tiles = (int)m_tiles;
  p.n_tiles = (int)n_tiles;
  {
    // N-tiles per rasterisation group: as many as keep the group's slice of B (all of K)
    // within about 32 MB of L2.  When K is so long that fewer than ~sqrt(CTA groups) tiles
    // fit, no slice stays resident anyway; the groups working at the same time then read the
    // least from DRAM with a near-square footprint (as many N-tiles as M-tiles), since each
    // distinct A row-block and B column-block they touch is fetched once per wave.  That
    // holds only where such a group has a wave's worth of tiles: with few M-tiles a wave
    // spans several groups and touches every A row-block whatever the width, and the L2
    // width measured faster (the weight gradients of a 2048-wide layer, 8 M-tiles and K =
    // 16384: dW_d 361 -> 348 us, dW_o 100.5 -> 98 us).
    const int64_t b_tile_bytes = (int64_t)var->un * row_bytes(W->dtype, K);
    int64_t gn = ((int64_t)32 << 20) / (b_tile_bytes > 0 ? b_tile_bytes : 1);
    int64_t square = 1;
    while ((square + 1) * (square + 1) <= d->sms / var->cg) ++square;
    if (gn < square && m_tiles * square >= d->sms / var->cg) gn = square;
    gn = gn < 1 ? 1 : (gn > n_tiles ? n_tiles : gn);
    p.group_n = (int)gn;
  }
  // Split-K for the linear fp32-output program when the tiles alone leave the last wave of
  // CTA groups mostly idle: the slices reduce-add into a zeroed output (fp32 adds in any
  // order: not bitwise reproducible from run to run).
  {
    const int64_t tiles = m_tiles * n_tiles;
    const int64_t groups = d->sms / var->cg;
    const int64_t num_kb = (K + var->bk - 1) / var->bk;
    int best = 1;
    double best_score = 0.0;
    // split only when a single pass leaves more than a quarter of the groups idle: the memset
    // and the reduce-adds cost more than the idle groups otherwise
    const double eff1 = (double)tiles / (double)(((tiles + groups - 1) / groups) * groups);
    if (epi == EPI_STORE && out->dtype == CODA_F32 && eff1 < 0.75) {
      const int64_t k_rows = (K + bk - 1) / bk;   // 128-byte rows of K: each slice keeps at least 32
      for (int sk = 1; sk <= 8; ++sk) {
        if (sk > 1 && k_rows / sk < 32) break;
        const int64_t work = tiles * sk;
        const double eff = (double)work / (double)(((work + groups - 1) / groups) * groups);
        const double score = eff - 0.02 * (sk - 1);
        if (score > best_score + 1e-9) {
          best_score = score;
          best = sk;
        }
      }
    }
    p.k_splits = best;
    p.kb_per_split = (int)((num_kb + best - 1) / best);
    if (best > 1) {
      const cudaStream_t cs = static_cast<cudaStream_t>(stream);
      const size_t row_bytes = (size_t)N * 4;
      const cudaError_t me = out->ld == N ? cudaMemsetAsync(out->ptr, 0, row_bytes * (size_t)M, cs)
                                          : cudaMemset2DAsync(out->ptr, (size_t)out->ld * 4, 0, row_bytes, (size_t)M, cs);
      if (me != cudaSuccess) return CODA_ERR_LAUNCH;
    }
  }
  p.flags = (has(CODA_OP_ROW_SUMSQ_PARTIAL) ? F_PARTIAL : 0) | (has(CODA_OP_AMAX) ? F_AMAX : 0) |
            (has(CODA_OP_COL_SCALE) || (epi == EPI_RMSBWD && sd.col_scale) ? F_COLSCALE : 0) |
            (has(CODA_OP_ROW_SCALE) ? F_ROWSCALE : 0) | (has(CODA_OP_COL_DOT_PARTIAL) ? F_COLPART : 0) |
            (epi == EPI_RMSBWD && !sd.aux_in2 ? F_NO_SIDE1 : 0);
  if (ab_ready && g_launch_overlap) p.flags |= F_AB_READY;
  // One group holds every N-tile, so each A row-block is read only by the CTA groups of one
  // wave, while all of B is reused by every wave.  With a long K, a wave streams more A than
  // L2 keeps beside B, and A at normal priority pushed B out (G3 of the block forward, K = 8192:
  // B re-read every wave, 537 MB read for 369 MB of compulsory reads).  There A is streamed
  // with evict_first (411 MB).  With K = 2048 the same policy measured slower, so it is kept
  // to long K, and to a B that L2 can hold (at most 48 MB).
  if (p.group_n == p.n_tiles && (K + bk - 1) / bk >= 128 &&
      n_tiles * (int64_t)var->un * row_bytes(W->dtype, K) <= ((int64_t)48 << 20))
    p.flags |= F_A_STREAM;
  switch (g_inject_once.exchange(0)) {
    case 1: p.flags |= F_INJECT_SKIP; break;
    case 2: p.flags |= F_INJECT_RANK1; break;
    case 3: p.flags |= F_INJECT_RANK0; break;
    default: break;
  }
  p.up_offset = (int)N;
  p.tensor_scale = has(CODA_OP_TENSOR_SCALE) ? sd.tensor_scale : 1.0f;
  p.out_scale = (out->dtype == CODA_E4M3 || epi == EPI_XENT_BWD) ? sd.out_scale : 1.0f;
  p.row_scale = sd.row_scale;
  p.row_coef = sd.row_coef;
  p.col_scale = sd.col_scale;
  p.rope_cos = sd.rope_cos;
  p.rope_sin = sd.rope_sin;
  p.rope_seq_len = sd.rope_seq_len > 0 ? sd.rope_seq_len : 1;
  p.rope_head_dim = sd.rope_head_dim;
  p.rope_ncols = has(CODA_OP_ROPE) ? sd.rope_ncols : 0;
  p.row_part = ax.row_partials;
  p.row_part_ld = ax.row_partials_ld;
  p.col_part = ax.col_partials;
  p.col_part_ld = ax.col_partials_ld;
  p.row_part2 = ax.row_partials2;
  p.row_out = ax.row_values;
  p.row_index = sd.row_index;
  p.amax = reinterpret_cast<unsigned int*>(ax.amax);
  p.fp4_scale = out->dtype == CODA_NVFP4 ? sd.out_fp4_scale : 1.0f;
  p.out_sf = reinterpret_cast<uint8_t*>(ax.out_block_scales);
  p.out_sf_kc = N / 64;
  p.status = d->status;
  p.timeout_ns = (unsigned long long)g_watchdog_ms * 1000000ull;
  L.sms = d->sms;
  L.overlap = g_launch_overlap;
  const cudaError_t e = var->fn(L, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CODA_OK : CODA_ERR_LAUNCH;
}

int coda_gemm_epilogue(const coda_tensor* A, const coda_tensor* W, const coda_epilogue_program* prog,
                       const coda_side_inputs* side, const coda_tensor* out, const coda_aux_outputs* aux,
                       void* stream) {
  return gemm_epilogue_impl(A, W, prog, side, out, aux, stream, false);
}

int coda_rms_partial_reduce(const float* partials, int64_t ld, int32_t nparts, int64_t M, int64_t d, float eps,
                            int32_t mode, const float* rowscale, float* out, void* stream) {
  if (!partials || !out) return CODA_ERR_NULL;
  if (mode != CODA_REDUCE_RSQRT_MEAN && mode != CODA_REDUCE_SCALE_SUM) return CODA_ERR_SHAPE;
  if (mode == CODA_REDUCE_SCALE_SUM && !rowscale) return CODA_ERR_NULL;
  if (M < 0 || d < 1 || nparts < 1 || ld < M) return CODA_ERR_SHAPE;
  if (M == 0) return CODA_OK;
  DevState* dv;
  int st = ensure_device(&dv);
  if (st != CODA_OK) return st;
  cudaError_t e = launch_partial_reduce(partials, ld, nparts, M, 1.0f / (float)d, eps, mode, rowscale, out,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CODA_OK : CODA_ERR_LAUNCH;
}

// coda_row_rms, also setting *zero (optional) to 0: the chains' amax reset, folded into the
// chain's first kernel so that no memset interrupts the launch overlap
static int row_rms_impl(const coda_tensor* X, float eps, float* r_out, void* stream, float* zero,
                        bool beside = false) {
  int st;
  if ((st = check_tensor(X, false)) != CODA_OK) return st;
  if (!r_out) return CODA_ERR_NULL;
  if (X->dtype != CODA_BF16) return CODA_ERR_DTYPE;
  if (X->cols < 1 || X->cols % 8 != 0) return CODA_ERR_SHAPE;
  if (X->rows == 0) return CODA_OK;
  DevState* dv;
  if ((st = ensure_device(&dv)) != CODA_OK) return st;
  cudaError_t e = launch_row_rms(X->ptr, X->rows, X->cols, X->ld, eps, r_out, static_cast<cudaStream_t>(stream),
                                 dv->sms, zero, beside);
  return e == cudaSuccess ? CODA_OK : CODA_ERR_LAUNCH;
}

int coda_row_rms(const coda_tensor* X, float eps, float* r_out, void* stream) {
  return row_rms_impl(X, eps, r_out, stream, nullptr);
}

int coda_quantize_e4m3(const coda_tensor* X, float scale, const coda_tensor* Q, float* amax, void* stream) {
  int st;
  if ((st = check_tensor(X, false)) != CODA_OK) return st;
  if ((st = check_tensor(Q, false)) != CODA_OK) return st;
  if (X->dtype != CODA_BF16 || Q->dtype != CODA_E4M3) return CODA_ERR_DTYPE;
  if (Q->rows != X->rows || Q->cols != X->cols || X->cols % 16 != 0) return CODA_ERR_SHAPE;
  if (!(scale > 0.f) || !(scale < INFINITY)) return CODA_ERR_SHAPE;
  if (X->rows == 0 || X->cols == 0) return CODA_OK;
  DevState* dv;
  if ((st = ensure_device(&dv)) != CODA_OK) return st;
  cudaError_t e = launch_quantize_e4m3(X->ptr, X->rows, X->cols, X->ld, 1.0f / scale, Q->ptr, Q->ld, amax,
                                       static_cast<cudaStream_t>(stream), dv->sms);
  return e == cudaSuccess ? CODA_OK : CODA_ERR_LAUNCH;
}

size_t coda_nvfp4_scale_bytes(int64_t R, int64_t K) {
  if (R <= 0 || K <= 0) return 0;
  return (size_t)((R + 127) / 128) * (size_t)(K / 64) * 512u;
}

int coda_quantize_nvfp4(const coda_tensor* X, float s, const coda_tensor* Q, void* block_scales, float* amax,
                        void* stream) {
  int st;
  if ((st = check_tensor(X, false)) != CODA_OK) return st;
  if ((st = check_tensor(Q, false)) != CODA_OK) return st;
  if (X->dtype != CODA_BF16 || Q->dtype != CODA_NVFP4) return CODA_ERR_DTYPE;
  if (Q->rows != X->rows || Q->cols != X->cols || X->cols % 64 != 0) return CODA_ERR_SHAPE;
  if (!(s > 0.f) || !(s < INFINITY)) return CODA_ERR_SHAPE;
  if (X->rows == 0 || X->cols == 0) return CODA_OK;
  if (!block_scales) return CODA_ERR_NULL;
  if (!aligned16(block_scales)) return CODA_ERR_ALIGN;
  DevState* dv;
  if ((st = ensure_device(&dv)) != CODA_OK) return st;
  cudaError_t e = launch_quantize_nvfp4(X->ptr, X->rows, X->cols, X->ld, s, Q->ptr, Q->ld / 2,
                                        static_cast<uint8_t*>(block_scales), amax,
                                        static_cast<cudaStream_t>(stream), dv->sms);
  return e == cudaSuccess ? CODA_OK : CODA_ERR_LAUNCH;
}

int coda_quantize_nvfp4_t(const coda_tensor* X, int32_t mode, float s, const coda_tensor* Q, void* block_scales,
                          const coda_tensor* Q_rows, void* row_block_scales, float* amax, void* stream) {
  int st;
  if ((st = check_tensor(X, false)) != CODA_OK) return st;
  if ((st = check_tensor(Q, false)) != CODA_OK) return st;
  if (X->dtype != CODA_BF16 || Q->dtype != CODA_NVFP4) return CODA_ERR_DTYPE;
  if (mode != CODA_QT_PLAIN && mode != CODA_QT_SWIGLU) return CODA_ERR_SHAPE;
  const int64_t R = X->rows, C = mode == CODA_QT_SWIGLU ? X->cols / 2 : X->cols;
  if (mode == CODA_QT_SWIGLU && X->cols % 2 != 0) return CODA_ERR_SHAPE;
  if (Q->rows != C || Q->cols != R || R % 64 != 0 || C % 128 != 0) return CODA_ERR_SHAPE;
  if (!(s > 0.f) || !(s < INFINITY)) return CODA_ERR_SHAPE;
  if (Q_rows) {
    if ((st = check_tensor(Q_rows, false)) != CODA_OK) return st;
    if (Q_rows->dtype != CODA_NVFP4) return CODA_ERR_DTYPE;
    if (Q_rows->rows != R || Q_rows->cols != C || R % 128 != 0) return CODA_ERR_SHAPE;
  }
  if (R == 0 || C == 0) return CODA_OK;
  if (!block_scales || (Q_rows && !row_block_scales)) return CODA_ERR_NULL;
  if (!aligned16(block_scales) || (Q_rows && !aligned16(row_block_scales))) return CODA_ERR_ALIGN;
  DevState* dv;
  if ((st = ensure_device(&dv)) != CODA_OK) return st;
  cudaError_t e = launch_quantize_nvfp4_t(X->ptr, R, C, X->ld, mode == CODA_QT_SWIGLU, s, Q->ptr, Q->ld / 2,
                                          static_cast<uint8_t*>(block_scales), Q_rows ? Q_rows->ptr : nullptr,
                                          Q_rows ? Q_rows->ld / 2 : 0, static_cast<uint8_t*>(row_block_scales), amax,
                                          static_cast<cudaStream_t>(stream), dv->sms);
  return e == cudaSuccess ? CODA_OK : CODA_ERR_LAUNCH;
}

int coda_col_reduce(const float* parts, int64_t nblocks, int64_t N, int64_t ld, float* out, void* stream) {
  if (!parts || !out) return CODA_ERR_NULL;
  if (nblocks < 0 || N < 0 || ld < N) return CODA_ERR_SHAPE;
  if (N == 0) return CODA_OK;
  DevState* dv;
  int st = ensure_device(&dv);
  if (st != CODA_OK) return st;
  cudaError_t e = launch_col_reduce(parts, nblocks, N, ld, out, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CODA_OK : CODA_ERR_LAUNCH;
}

int coda_fold_gain(const coda_tensor* W, const float* g, float out_scale, const coda_tensor* W_out, void* stream) {
  int st;
  if ((st = check_tensor(W, false)) != CODA_OK) return st;
  if ((st = check_tensor(W_out, false)) != CODA_OK) return st;
  if (!g) return CODA_ERR_NULL;
  if (!aligned16(g)) return CODA_ERR_ALIGN;
  if (W->layout != CODA_ROW_MAJOR || W_out->layout != CODA_ROW_MAJOR) return CODA_ERR_SHAPE;
  int kind;
  if (W->dtype == CODA_F32 && W_out->dtype == CODA_F32) kind = FOLD_OUT_F32;
  else if (W->dtype == CODA_BF16 && W_out->dtype == CODA_BF16) kind = FOLD_OUT_BF16;
  else if (W->dtype == CODA_BF16 && W_out->dtype == CODA_E4M3) kind = FOLD_OUT_E4M3;
  else return CODA_ERR_DTYPE;
  if (!(out_scale > 0.0f) || !(out_scale < INFINITY)) return CODA_ERR_SHAPE;
  if (kind == FOLD_OUT_E4M3 && W->ptr == W_out->ptr) return CODA_ERR_SHAPE;   // widths differ: no in place
  const int vec = kind == FOLD_OUT_F32 ? 4 : kind == FOLD_OUT_E4M3 ? 16 : 8;
  if (W->rows != W_out->rows || W->cols != W_out->cols || W->cols % vec != 0) return CODA_ERR_SHAPE;
  if (W->rows == 0 || W->cols == 0) return CODA_OK;
  DevState* dv;
  if ((st = ensure_device(&dv)) != CODA_OK) return st;
  cudaError_t e = launch_fold_gain(W->ptr, W->rows, W->cols, W->ld, g, 1.0f / out_scale, W_out->ptr, W_out->ld,
                                   kind, static_cast<cudaStream_t>(stream), dv->sms);
  return e == cudaSuccess ? CODA_OK : CODA_ERR_LAUNCH;
}

int coda_rope_table(int32_t seq_len, int32_t head_dim, double base, float* cos_out, float* sin_out, void* stream) {
  if (!cos_out || !sin_out) return CODA_ERR_NULL;
  if (seq_len < 1 || head_dim < 2 || head_dim % 2 != 0 || !(base > 0.0)) return CODA_ERR_SHAPE;
  DevState* dv;
  int st = ensure_device(&dv);
  if (st != CODA_OK) return st;
  cudaError_t e = launch_rope_table(seq_len, head_dim, base, cos_out, sin_out, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CODA_OK : CODA_ERR_LAUNCH;
}

int coda_rms_gain(const coda_tensor* X, const float* g, float eps, float* r_out, const coda_tensor* u_out,
                  void* stream) {
  int st;
  if ((st = check_tensor(X, false)) != CODA_OK) return st;
  if ((st = check_tensor(u_out, false)) != CODA_OK) return st;
  if (!r_out || !g) return CODA_ERR_NULL;
  if (!aligned16(g)) return CODA_ERR_ALIGN;
  if (X->dtype != CODA_BF16 || u_out->dtype != CODA_BF16) return CODA_ERR_DTYPE;
  if (X->cols < 1 || X->cols % 8 != 0 || u_out->rows != X->rows || u_out->cols != X->cols) return CODA_ERR_SHAPE;
  if (X->rows == 0) return CODA_OK;
  DevState* dv;
  if ((st = ensure_device(&dv)) != CODA_OK) return st;
  cudaError_t e = launch_rms_gain(X->ptr, X->rows, X->cols, X->ld, g, eps, r_out, u_out->ptr, u_out->ld,
                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CODA_OK : CODA_ERR_LAUNCH;
}

int coda_xent_combine(const float* Pm, const float* Ps, int64_t ld, int32_t nparts, int64_t M,
                      const float* target_logit, const int32_t* targets, int64_t V, float* lse, float* loss,
                      float* mean, void* stream) {
  if (!Pm || !Ps || !target_logit || !targets || !lse || !loss) return CODA_ERR_NULL;
  if (M < 0 || nparts < 1 || ld < M || V < 1) return CODA_ERR_SHAPE;
  if (M == 0) return CODA_OK;
  DevState* dv;
  int st = ensure_device(&dv);
  if (st != CODA_OK) return st;
  cudaError_t e = launch_xent_reduce(Pm, Ps, ld, nparts, M, target_logit, targets, V, lse, loss, mean,
                                     static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CODA_OK : CODA_ERR_LAUNCH;
}

size_t coda_workspace_size(int32_t which, int64_t M, int64_t H, int64_t F) {
  if (M < 0 || H < 0 || F < 0) return 0;
  if (which == CODA_WS_BLOCK_FWD) return (size_t)((H + 255) / 256) * (size_t)M * sizeof(float);
  if (which == CODA_WS_BLOCK_BWD || which == CODA_WS_XENT_BWD)
    return ((size_t)((F + 255) / 256) * (size_t)M + (size_t)((M + 31) / 32) * (size_t)H) * sizeof(float);
  if (which == CODA_WS_XENT_FWD) return (size_t)(2 * ((F + 255) / 256) + 1) * (size_t)M * sizeof(float);
  if (which == CODA_WS_MLP_FP8_BWD) return (size_t)((F + 255) / 256) * (size_t)M * sizeof(float);
  if (which == CODA_WS_MLP_NVFP4_BWD) return (size_t)((F + 127) / 128) * (size_t)M * sizeof(float);
  return 0;
}

}  // extern "C"

// ------------------------------------------------------------------- chains
namespace {
coda_tensor mk(const void* p, int dt, int64_t rows, int64_t cols, int64_t ld, int layout = CODA_ROW_MAJOR) {
  coda_tensor t;
  t.ptr = const_cast<void*>(p);
  t.dtype = dt;
  t.layout = layout;
  t.rows = rows;
  t.cols = cols;
  t.ld = ld;
  return t;
}
coda_epilogue_program prog_of(std::initializer_list<int> ops) {
  coda_epilogue_program p{};
  for (int o : ops) p.ops[p.n_ops++] = o;
  return p;
}
}  // namespace

extern "C" {

int coda_block_forward(const coda_block_fwd* io, void* stream) {
  if (!io) return CODA_ERR_NULL;
  const int64_t M = io->M, H = io->H, F = io->F;
  if (M < 0 || H < 32 || F < 128 || H % 32 != 0 || F % 128 != 0) return CODA_ERR_SHAPE;
  if (!io->O || !io->R || !io->W_o || !io->W_gu || !io->W_d || !io->h || !io->r || !io->a || !io->Y ||
      !io->workspace)
    return CODA_ERR_NULL;
  const bool broadcast_gain = io->g != nullptr;
  if (broadcast_gain && !io->u) return CODA_ERR_NULL;
  if (M == 0) return CODA_OK;
  int st;
  const int64_t nparts = (H + 255) / 256;
  // G1: h = O W_o^T + R, partial sums of squares of h [, u = h * g]
  {
    coda_tensor A = mk(io->O, CODA_BF16, M, H, H), W = mk(io->W_o, CODA_BF16, H, H, H);
    coda_tensor R = mk(io->R, CODA_BF16, M, H, H), out = mk(io->h, CODA_BF16, M, H, H);
    coda_tensor U = mk(io->u, CODA_BF16, M, H, H);
    coda_epilogue_program pg =
        broadcast_gain ? prog_of({CODA_OP_ADD_SIDE, CODA_OP_ROW_SUMSQ_PARTIAL, CODA_OP_STORE_COL_SCALED})
                       : prog_of({CODA_OP_ADD_SIDE, CODA_OP_ROW_SUMSQ_PARTIAL});
    coda_side_inputs sd{};
    sd.residual = &R;
    sd.col_scale = io->g;
    coda_aux_outputs ax{};
    ax.row_partials = io->workspace;
    ax.row_partials_ld = M;
    ax.store_aux = broadcast_gain ? &U : nullptr;
    if ((st = coda_gemm_epilogue(&A, &W, &pg, &sd, &out, &ax, stream)) != CODA_OK) return st;
  }
  // r = 1 / sqrt(sum of partials / H + eps)
  if ((st = coda_rms_partial_reduce(io->workspace, M, (int32_t)nparts, M, H, io->eps, CODA_REDUCE_RSQRT_MEAN, nullptr,
                                    io->r, stream)) != CODA_OK)
    return st;
  // G2: [G | U] = r (u W_gu^T) (or r (h W_gu'^T));  a = silu(G) U  [+ saved Z]
  {
    coda_tensor A = mk(broadcast_gain ? io->u : io->h, CODA_BF16, M, H, H);
    coda_tensor W = mk(io->W_gu, CODA_BF16, 2 * F, H, H);
    coda_tensor out = mk(io->a, CODA_BF16, M, F, F);
    coda_tensor Z = mk(io->Z, CODA_BF16, M, 2 * F, 2 * F);
    coda_epilogue_program pg = io->Z ? prog_of({CODA_OP_ROW_SCALE, CODA_OP_STORE_AUX, CODA_OP_SWIGLU})
                                     : prog_of({CODA_OP_ROW_SCALE, CODA_OP_SWIGLU});
    coda_side_inputs sd{};
    sd.row_scale = io->r;
    coda_aux_outputs ax{};
    ax.store_aux = io->Z ? &Z : nullptr;
    if ((st = gemm_epilogue_impl(&A, &W, &pg, &sd, &out, &ax, stream, true)) != CODA_OK) return st;
  }
  // G3: Y = a W_d^T + h  [+ partial sums of squares of Y for the next layer]
  {
    coda_tensor A = mk(io->a, CODA_BF16, M, F, F), W = mk(io->W_d, CODA_BF16, H, F, F);
    coda_tensor R = mk(io->h, CODA_BF16, M, H, H), out = mk(io->Y, CODA_BF16, M, H, H);
    coda_epilogue_program pg = io->Y_partials ? prog_of({CODA_OP_ADD_SIDE, CODA_OP_ROW_SUMSQ_PARTIAL})
                                              : prog_of({CODA_OP_ADD_SIDE});
    coda_side_inputs sd{};
    sd.residual = &R;
    coda_aux_outputs ax{};
    ax.row_partials = io->Y_partials;
    ax.row_partials_ld = M;
    if ((st = coda_gemm_epilogue(&A, &W, &pg, &sd, &out, &ax, stream)) != CODA_OK) return st;
  }
  return CODA_OK;
}

int coda_block_backward(const coda_block_bwd* io, void* stream) {
  if (!io) return CODA_ERR_NULL;
  const int64_t M = io->M, H = io->H, F = io->F;
  if (M < 0 || H < 32 || F < 128 || H % 32 != 0 || F % 128 != 0) return CODA_ERR_SHAPE;
  if (!io->O || !io->W_o || !io->W_gu || !io->W_d || !io->g || !io->h || !io->r || !io->Z || !io->a || !io->dY ||
      !io->e || !io->dh || !io->dO || !io->dW_o || !io->dW_gu || !io->dW_d || !io->dg || !io->c || !io->workspace)
    return CODA_ERR_NULL;
  if (M == 0) return CODA_OK;
  int st;
  float* S = io->workspace;                          // [F/256, M] row partials of e . Z
  float* Dg = io->workspace + ((F + 255) / 256) * M; // [ceil(M/32), H] column partials of h t
  const int64_t nS = (F + 255) / 256;
  const int64_t nDg = (M + 31) / 32;
  // b1: e = r [dA U silu'(G) | dA silu(G)],  dA = dY W_d;  row partials of e . Z
  {
    coda_tensor A = mk(io->dY, CODA_BF16, M, H, H);
    coda_tensor W = mk(io->W_d, CODA_BF16, F, H, F, CODA_COL_MAJOR);  // logical W_d^T
    coda_tensor Z = mk(io->Z, CODA_BF16, M, 2 * F, 2 * F), out = mk(io->e, CODA_BF16, M, 2 * F, 2 * F);
    coda_epilogue_program pg = prog_of({CODA_OP_SWIGLU_BWD, CODA_OP_ROW_SCALE, CODA_OP_ROW_DOT_PARTIAL});
    coda_side_inputs sd{};
    sd.aux_in = &Z;
    sd.row_scale = io->r;
    coda_aux_outputs ax{};
    ax.row_partials = S;
    ax.row_partials_ld = M;
    if ((st = coda_gemm_epilogue(&A, &W, &pg, &sd, &out, &ax, stream)) != CODA_OK) return st;
  }
  // b2: dW_d = dY^T a
  {
    coda_tensor A = mk(io->dY, CODA_BF16, H, M, H, CODA_COL_MAJOR), W = mk(io->a, CODA_BF16, F, M, F, CODA_COL_MAJOR);
    coda_tensor out = mk(io->dW_d, CODA_F32, H, F, F);
    coda_epilogue_program pg = prog_of({});
    if ((st = gemm_epilogue_impl(&A, &W, &pg, nullptr, &out, nullptr, stream, true)) != CODA_OK) return st;
  }
  // b3: c = r * sum(S) / H
  if ((st = coda_rms_partial_reduce(S, M, (int32_t)nS, M, H, 0.f, CODA_REDUCE_SCALE_SUM, io->r, io->c, stream)) !=
      CODA_OK)
    return st;
  // b4: t = e W_gu;  dh = g t - c h + dY;  column partials of h t
  {
    coda_tensor A = mk(io->e, CODA_BF16, M, 2 * F, 2 * F);
    coda_tensor W = mk(io->W_gu, CODA_BF16, H, 2 * F, H, CODA_COL_MAJOR);  // logical W_gu^T
    coda_tensor h = mk(io->h, CODA_BF16, M, H, H), dY = mk(io->dY, CODA_BF16, M, H, H);
    coda_tensor out = mk(io->dh, CODA_BF16, M, H, H);
    coda_epilogue_program pg = prog_of({CODA_OP_RMSBWD_COMBINE, CODA_OP_COL_DOT_PARTIAL});
    coda_side_inputs sd{};
    sd.aux_in = &h;
    sd.aux_in2 = &dY;
    sd.col_scale = io->g;
    sd.row_coef = io->c;
    coda_aux_outputs ax{};
    ax.col_partials = Dg;
    ax.col_partials_ld = H;
    if ((st = gemm_epilogue_impl(&A, &W, &pg, &sd, &out, &ax, stream, true)) != CODA_OK) return st;
  }
  // b5: dg = column sums of the partials
  if ((st = coda_col_reduce(Dg, nDg, H, H, io->dg, stream)) != CODA_OK) return st;
  // b6: dW_gu[n, k] = g_k (e^T h)[n, k]
  {
    coda_tensor A = mk(io->e, CODA_BF16, 2 * F, M, 2 * F, CODA_COL_MAJOR);
    coda_tensor W = mk(io->h, CODA_BF16, H, M, H, CODA_COL_MAJOR);
    coda_tensor out = mk(io->dW_gu, CODA_F32, 2 * F, H, H);
    coda_epilogue_program pg = prog_of({CODA_OP_COL_SCALE});
    coda_side_inputs sd{};
    sd.col_scale = io->g;
    if ((st = gemm_epilogue_impl(&A, &W, &pg, &sd, &out, nullptr, stream, true)) != CODA_OK) return st;
  }
  // b7: dO = dh W_o
  {
    coda_tensor A = mk(io->dh, CODA_BF16, M, H, H);
    coda_tensor W = mk(io->W_o, CODA_BF16, H, H, H, CODA_COL_MAJOR);  // logical W_o^T
    coda_tensor out = mk(io->dO, CODA_BF16, M, H, H);
    coda_epilogue_program pg = prog_of({});
    if ((st = gemm_epilogue_impl(&A, &W, &pg, nullptr, &out, nullptr, stream, true)) != CODA_OK) return st;
  }
  // b8: dW_o = dh^T O
  {
    coda_tensor A = mk(io->dh, CODA_BF16, H, M, H, CODA_COL_MAJOR), W = mk(io->O, CODA_BF16, H, M, H, CODA_COL_MAJOR);
    coda_tensor out = mk(io->dW_o, CODA_F32, H, H, H);
    coda_epilogue_program pg = prog_of({});
    if ((st = gemm_epilogue_impl(&A, &W, &pg, nullptr, &out, nullptr, stream, true)) != CODA_OK) return st;
  }
  return CODA_OK;
}

int coda_lm_head_xent_forward(const coda_lm_head_xent_io* io, void* stream) {
  if (!io) return CODA_ERR_NULL;
  if (!io->h || !io->g || !io->W_v || !io->targets || !io->u || !io->r || !io->lse || !io->loss || !io->loss_mean ||
      !io->workspace)
    return CODA_ERR_NULL;
  const int64_t M = io->M, H = io->H, V = io->V;
  if (M < 0 || H < 8 || H % 8 != 0 || V < 32 || V % 32 != 0) return CODA_ERR_SHAPE;
  if (M == 0) return CODA_OK;
  int st;
  const int64_t np = (V + 255) / 256;
  float* Pm = io->workspace;
  float* Ps = io->workspace + np * M;
  float* T = io->workspace + 2 * np * M;
  coda_tensor h = mk(io->h, CODA_BF16, M, H, H), u = mk(io->u, CODA_BF16, M, H, H);
  if ((st = coda_rms_gain(&h, io->g, io->eps, io->r, &u, stream)) != CODA_OK) return st;
  {
    coda_tensor W = mk(io->W_v, CODA_BF16, V, H, H), z = mk(nullptr, CODA_BF16, M, V, V);
    coda_epilogue_program pg = prog_of({CODA_OP_ROW_SCALE, CODA_OP_XENT_PARTIAL});
    coda_side_inputs sd{};
    sd.row_scale = io->r;
    sd.row_index = io->targets;
    coda_aux_outputs ax{};
    ax.row_partials = Pm;
    ax.row_partials2 = Ps;
    ax.row_partials_ld = M;
    ax.row_values = T;
    if ((st = coda_gemm_epilogue(&u, &W, &pg, &sd, &z, &ax, stream)) != CODA_OK) return st;
  }
  return coda_xent_combine(Pm, Ps, M, (int32_t)np, M, T, io->targets, V, io->lse, io->loss, io->loss_mean, stream);
}

int coda_lm_head_xent_backward(const coda_lm_head_xent_bwd_io* io, void* stream) {
  if (!io) return CODA_ERR_NULL;
  if (!io->h || !io->g || !io->W_v || !io->targets || !io->u || !io->r || !io->lse || !io->e || !io->dh ||
      !io->dW_v || !io->dg || !io->c || !io->workspace)
    return CODA_ERR_NULL;
  const int64_t M = io->M, H = io->H, V = io->V;
  if (M < 0 || H < 32 || H % 32 != 0 || V < 32 || V % 32 != 0) return CODA_ERR_SHAPE;
  if (M == 0) return CODA_OK;
  int st;
  const int64_t np = (V + 255) / 256;
  float* S = io->workspace;              // [np, M] row partials of e . z
  float* Dg = io->workspace + np * M;    // [ceil(M/32), H] column partials of h t
  coda_tensor u = mk(io->u, CODA_BF16, M, H, H), e = mk(io->e, CODA_BF16, M, V, V);
  // e = r dloss (softmax - onehot) / M, logits recomputed; row partials of e . z
  {
    coda_tensor W = mk(io->W_v, CODA_BF16, V, H, H);
    coda_epilogue_program pg = prog_of({CODA_OP_ROW_SCALE, CODA_OP_XENT_BWD, CODA_OP_ROW_DOT_PARTIAL});
    coda_side_inputs sd{};
    sd.row_scale = io->r;
    sd.row_coef = io->lse;
    sd.row_index = io->targets;
    sd.out_scale = io->dloss / (float)M;
    coda_aux_outputs ax{};
    ax.row_partials = S;
    ax.row_partials_ld = M;
    if ((st = coda_gemm_epilogue(&u, &W, &pg, &sd, &e, &ax, stream)) != CODA_OK) return st;
  }
  // c = r s / H
  if ((st = coda_rms_partial_reduce(S, M, (int32_t)np, M, H, 0.f, CODA_REDUCE_SCALE_SUM, io->r, io->c, stream)) !=
      CODA_OK)
    return st;
  // t = e W_v;  dh = g t - c h;  column partials of h t
  {
    coda_tensor W = mk(io->W_v, CODA_BF16, H, V, H, CODA_COL_MAJOR);   // logical W_v^T
    coda_tensor h = mk(io->h, CODA_BF16, M, H, H), out = mk(io->dh, CODA_BF16, M, H, H);
    coda_epilogue_program pg = prog_of({CODA_OP_RMSBWD_COMBINE, CODA_OP_COL_DOT_PARTIAL});
    coda_side_inputs sd{};
    sd.aux_in = &h;
    sd.col_scale = io->g;
    sd.row_coef = io->c;
    coda_aux_outputs ax{};
    ax.col_partials = Dg;
    ax.col_partials_ld = H;
    if ((st = gemm_epilogue_impl(&e, &W, &pg, &sd, &out, &ax, stream, true)) != CODA_OK) return st;
  }
  if ((st = coda_col_reduce(Dg, (M + 31) / 32, H, H, io->dg, stream)) != CODA_OK) return st;
  // dW_v = e^T u
  {
    coda_tensor A = mk(io->e, CODA_BF16, V, M, V, CODA_COL_MAJOR), W = mk(io->u, CODA_BF16, H, M, H, CODA_COL_MAJOR);
    coda_tensor out = mk(io->dW_v, CODA_F32, V, H, H);
    coda_epilogue_program pg = prog_of({});
    if ((st = gemm_epilogue_impl(&A, &W, &pg, nullptr, &out, nullptr, stream, true)) != CODA_OK) return st;
  }
  return CODA_OK;
}

int coda_rope_backward(const coda_tensor* dout, const coda_tensor* out, const float* r, const float* rope_cos,
                       const float* rope_sin, int32_t seq_len, int32_t head_dim, int32_t rope_ncols, int64_t H,
                       const coda_tensor* e_out, float* c_out, void* stream) {
  int st;
  if ((st = check_tensor(dout, false)) != CODA_OK) return st;
  if ((st = check_tensor(out, false)) != CODA_OK) return st;
  if ((st = check_tensor(e_out, false)) != CODA_OK) return st;
  if (!r || !rope_cos || !rope_sin || !c_out) return CODA_ERR_NULL;
  if (!aligned16(rope_cos) || !aligned16(rope_sin)) return CODA_ERR_ALIGN;
  if (dout->dtype != CODA_BF16 || out->dtype != CODA_BF16 || e_out->dtype != CODA_BF16) return CODA_ERR_DTYPE;
  const int64_t M = dout->rows, N = dout->cols;
  if (out->rows != M || out->cols != N || e_out->rows != M || e_out->cols != N || out->ld != dout->ld) return CODA_ERR_SHAPE;
  if (N % 8 != 0 || head_dim < 8 || head_dim % 8 != 0 || rope_ncols < 0 || rope_ncols % head_dim != 0 ||
      rope_ncols > N || seq_len < 1 || H < 1)
    return CODA_ERR_SHAPE;
  if (M == 0) return CODA_OK;
  DevState* dv;
  if ((st = ensure_device(&dv)) != CODA_OK) return st;
  cudaError_t e = launch_rope_bwd(dout->ptr, out->ptr, M, N, dout->ld, r, rope_cos, rope_sin, seq_len, head_dim,
                                  rope_ncols, H, e_out->ptr, e_out->ld, c_out, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CODA_OK : CODA_ERR_LAUNCH;
}

int coda_qkv_rope_backward(const coda_qkv_rope_bwd_io* io, void* stream) {
  if (!io) return CODA_ERR_NULL;
  if (!io->h || !io->g || !io->W_qkv || !io->r || !io->out || !io->dout || !io->rope_cos || !io->rope_sin ||
      !io->e || !io->dh || !io->dW_qkv || !io->dg || !io->c || !io->workspace)
    return CODA_ERR_NULL;
  const int64_t M = io->M, H = io->H, N = io->N;
  if (M < 0 || H < 32 || H % 32 != 0 || N < 32 || N % 32 != 0) return CODA_ERR_SHAPE;
  if (M == 0) return CODA_OK;
  int st;
  coda_tensor dout = mk(io->dout, CODA_BF16, M, N, N), out = mk(io->out, CODA_BF16, M, N, N);
  coda_tensor e = mk(io->e, CODA_BF16, M, N, N);
  if ((st = coda_rope_backward(&dout, &out, io->r, io->rope_cos, io->rope_sin, io->seq_len, io->head_dim,
                               io->rope_ncols, H, &e, io->c, stream)) != CODA_OK)
    return st;
  float* Dg = io->workspace;
  {
    coda_tensor W = mk(io->W_qkv, CODA_BF16, H, N, H, CODA_COL_MAJOR);   // logical W_qkv^T
    coda_tensor h = mk(io->h, CODA_BF16, M, H, H), dres = mk(io->dres, CODA_BF16, M, H, H);
    coda_tensor dh = mk(io->dh, CODA_BF16, M, H, H);
    coda_epilogue_program pg = prog_of({CODA_OP_RMSBWD_COMBINE, CODA_OP_COL_DOT_PARTIAL});
    coda_side_inputs sd{};
    sd.aux_in = &h;
    sd.aux_in2 = io->dres ? &dres : nullptr;
    sd.col_scale = io->g;
    sd.row_coef = io->c;
    coda_aux_outputs ax{};
    ax.col_partials = Dg;
    ax.col_partials_ld = H;
    if ((st = coda_gemm_epilogue(&e, &W, &pg, &sd, &dh, &ax, stream)) != CODA_OK) return st;
  }
  if ((st = coda_col_reduce(Dg, (M + 31) / 32, H, H, io->dg, stream)) != CODA_OK) return st;
  {
    coda_tensor A = mk(io->e, CODA_BF16, N, M, N, CODA_COL_MAJOR), W = mk(io->h, CODA_BF16, H, M, H, CODA_COL_MAJOR);
    coda_tensor dW = mk(io->dW_qkv, CODA_F32, N, H, H);
    coda_epilogue_program pg = prog_of({CODA_OP_COL_SCALE});
    coda_side_inputs sd{};
    sd.col_scale = io->g;
    if ((st = gemm_epilogue_impl(&A, &W, &pg, &sd, &dW, nullptr, stream, true)) != CODA_OK) return st;
  }
  return CODA_OK;
}

int coda_qkv_rope(const coda_qkv_rope_io* io, void* stream) {
  if (!io) return CODA_ERR_NULL;
  if (!io->h || !io->W_qkv || !io->rope_cos || !io->rope_sin || !io->r || !io->out) return CODA_ERR_NULL;
  const int64_t M = io->M, H = io->H, N = io->N;
  if (M < 0 || H < 8 || N < 32 || io->seq_len < 1) return CODA_ERR_SHAPE;
  if (M == 0) return CODA_OK;
  int st;
  coda_tensor h = mk(io->h, CODA_BF16, M, H, H);
  // the QKV GEMM reads r only in its epilogue and its CTAs fit beside the pass
  if ((st = row_rms_impl(&h, io->eps, io->r, stream, nullptr, true)) != CODA_OK) return st;
  coda_tensor W = mk(io->W_qkv, CODA_BF16, N, H, H), out = mk(io->out, CODA_BF16, M, N, N);
  coda_epilogue_program pg = prog_of({CODA_OP_ROW_SCALE, CODA_OP_ROPE});
  coda_side_inputs sd{};
  sd.row_scale = io->r;
  sd.rope_cos = io->rope_cos;
  sd.rope_sin = io->rope_sin;
  sd.rope_seq_len = io->seq_len;
  sd.rope_head_dim = io->head_dim;
  sd.rope_ncols = io->rope_ncols;
  return gemm_epilogue_impl(&h, &W, &pg, &sd, &out, nullptr, stream, true);
}

int coda_mlp_fp8(const coda_mlp_fp8_io* io, void* stream) {
  if (!io) return CODA_ERR_NULL;
  if (!io->h || !io->X_q || !io->W_q || !io->W_dq || !io->r || !io->a_q || !io->amax || !io->Y || !io->Y_partials)
    return CODA_ERR_NULL;
  const int64_t M = io->M, H = io->H, F = io->F;
  if (M < 0 || H < 32 || F < 128 || H % 32 != 0 || F % 128 != 0) return CODA_ERR_SHAPE;
  if (!(io->s_a > 0.f)) return CODA_ERR_SHAPE;
  if (M == 0) return CODA_OK;
  int st;
  coda_tensor h = mk(io->h, CODA_BF16, M, H, H);
  // also amax = 0; the e4m3 gate/up GEMM reads r only in its epilogue and fits beside the pass
  if ((st = row_rms_impl(&h, io->eps, io->r, stream, io->amax, true)) != CODA_OK) return st;
  {
    coda_tensor A = mk(io->X_q, CODA_E4M3, M, H, H), W = mk(io->W_q, CODA_E4M3, 2 * F, H, H);
    coda_tensor out = mk(io->a_q, CODA_E4M3, M, F, F);
    coda_tensor Z = mk(io->Z, CODA_BF16, M, 2 * F, 2 * F);
    coda_epilogue_program pg =
        io->Z ? prog_of({CODA_OP_TENSOR_SCALE, CODA_OP_ROW_SCALE, CODA_OP_STORE_AUX, CODA_OP_SWIGLU, CODA_OP_AMAX})
              : prog_of({CODA_OP_TENSOR_SCALE, CODA_OP_ROW_SCALE, CODA_OP_SWIGLU, CODA_OP_AMAX});
    coda_side_inputs sd{};
    sd.tensor_scale = io->s_x * io->s_w;
    sd.row_scale = io->r;
    sd.out_scale = 1.0f / io->s_a;
    coda_aux_outputs ax{};
    ax.amax = io->amax;
    if (io->Z) ax.store_aux = &Z;
    if ((st = gemm_epilogue_impl(&A, &W, &pg, &sd, &out, &ax, stream, true)) != CODA_OK) return st;
  }
  {
    coda_tensor A = mk(io->a_q, CODA_E4M3, M, F, F), W = mk(io->W_dq, CODA_E4M3, H, F, F);
    coda_tensor out = mk(io->Y, CODA_BF16, M, H, H);
    coda_epilogue_program pg = prog_of({CODA_OP_TENSOR_SCALE, CODA_OP_ADD_SIDE, CODA_OP_ROW_SUMSQ_PARTIAL});
    coda_side_inputs sd{};
    sd.tensor_scale = io->s_a * io->s_wd;
    sd.residual = &h;
    coda_aux_outputs ax{};
    ax.row_partials = io->Y_partials;
    ax.row_partials_ld = M;
    if ((st = coda_gemm_epilogue(&A, &W, &pg, &sd, &out, &ax, stream)) != CODA_OK) return st;
  }
  return CODA_OK;
}

int coda_mlp_nvfp4(const coda_mlp_nvfp4_io* io, void* stream) {
  if (!io) return CODA_ERR_NULL;
  if (!io->h || !io->X_q || !io->X_sf || !io->W_q || !io->W_sf || !io->W_dq || !io->W_dsf || !io->r || !io->a_q ||
      !io->a_sf || !io->amax || !io->Y || !io->Y_partials)
    return CODA_ERR_NULL;
  const int64_t M = io->M, H = io->H, F = io->F;
  if (M < 0 || H < 256 || F < 256 || H % 256 != 0 || F % 256 != 0) return CODA_ERR_SHAPE;
  if (!(io->s_a > 0.f)) return CODA_ERR_SHAPE;
  if (M == 0) return CODA_OK;
  int st;
  coda_tensor h = mk(io->h, CODA_BF16, M, H, H);
  // also amax = 0; the many-CTA pass: the NVFP4 GEMM (ten warps of 168 registers) cannot sit
  // beside a resident one
  if ((st = row_rms_impl(&h, io->eps, io->r, stream, io->amax)) != CODA_OK) return st;
  {
    coda_tensor A = mk(io->X_q, CODA_NVFP4, M, H, H), W = mk(io->W_q, CODA_NVFP4, 2 * F, H, H);
    coda_tensor out = mk(io->a_q, CODA_NVFP4, M, F, F);
    coda_epilogue_program pg =
        prog_of({CODA_OP_TENSOR_SCALE, CODA_OP_ROW_SCALE, CODA_OP_SWIGLU, CODA_OP_AMAX});
    coda_side_inputs sd{};
    sd.tensor_scale = io->s_x * io->s_w;
    sd.row_scale = io->r;
    sd.a_block_scales = io->X_sf;
    sd.w_block_scales = io->W_sf;
    sd.out_fp4_scale = io->s_a;
    coda_aux_outputs ax{};
    ax.amax = io->amax;
    ax.out_block_scales = io->a_sf;
    if ((st = gemm_epilogue_impl(&A, &W, &pg, &sd, &out, &ax, stream, true)) != CODA_OK) return st;
  }
  {
    coda_tensor A = mk(io->a_q, CODA_NVFP4, M, F, F), W = mk(io->W_dq, CODA_NVFP4, H, F, F);
    coda_tensor out = mk(io->Y, CODA_BF16, M, H, H);
    coda_epilogue_program pg = prog_of({CODA_OP_TENSOR_SCALE, CODA_OP_ADD_SIDE, CODA_OP_ROW_SUMSQ_PARTIAL});
    coda_side_inputs sd{};
    sd.tensor_scale = io->s_a * io->s_wd;
    sd.residual = &h;
    sd.a_block_scales = io->a_sf;
    sd.w_block_scales = io->W_dsf;
    coda_aux_outputs ax{};
    ax.row_partials = io->Y_partials;
    ax.row_partials_ld = M;
    if ((st = coda_gemm_epilogue(&A, &W, &pg, &sd, &out, &ax, stream)) != CODA_OK) return st;
  }
  return CODA_OK;
}

int coda_mlp_fp8_backward(const coda_mlp_fp8_bwd_io* io, void* stream) {
  if (!io) return CODA_ERR_NULL;
  const int64_t M = io->M, H = io->H, F = io->F;
  if (M < 0 || H < 32 || F < 128 || H % 32 != 0 || F % 128 != 0) return CODA_ERR_SHAPE;
  if (!(io->s_x > 0.f) || !(io->s_w > 0.f) || !(io->s_wd > 0.f) || !(io->s_a > 0.f) || !(io->s_dy > 0.f) ||
      !(io->s_e > 0.f))
    return CODA_ERR_SHAPE;
  if (!io->W_q || !io->W_dq || !io->amax_dy || !io->amax_e || !io->dW_d || !io->dW) return CODA_ERR_NULL;
  if (M > 0 && (!io->h || !io->X_q || !io->Z || !io->a_q || !io->r || !io->dY || !io->dY_q || !io->e_q || !io->c ||
                !io->dh || !io->workspace))
    return CODA_ERR_NULL;
  if (M > 0 && !aligned16(io->workspace)) return CODA_ERR_ALIGN;
  int st;
  DevState* dv;
  if ((st = ensure_device(&dv)) != CODA_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(io->amax_dy, 0, sizeof(float), cs) != cudaSuccess ||
      cudaMemsetAsync(io->amax_e, 0, sizeof(float), cs) != cudaSuccess)
    return CODA_ERR_LAUNCH;
  if (M == 0) {   // sums over an empty batch: zero weight gradients
    if (cudaMemsetAsync(io->dW_d, 0, (size_t)H * F * sizeof(float), cs) != cudaSuccess ||
        cudaMemsetAsync(io->dW, 0, (size_t)2 * F * H * sizeof(float), cs) != cudaSuccess)
      return CODA_ERR_LAUNCH;
    return CODA_OK;
  }
  coda_tensor dY = mk(io->dY, CODA_BF16, M, H, H), dYq = mk(io->dY_q, CODA_E4M3, M, H, H);
  if ((st = coda_quantize_e4m3(&dY, io->s_dy, &dYq, io->amax_dy, stream)) != CODA_OK) return st;
  float* spart = io->workspace;   // [ceil(F / 256), M] row partials of sum e . Z
  {
    // dA = s_dy s_wd (dY_q W_dq); SwiGLU backward with r; e stored as e4m3, row partials
    coda_tensor W = mk(io->W_dq, CODA_E4M3, F, H, F, CODA_COL_MAJOR);   // logical W_d^T
    coda_tensor Z = mk(io->Z, CODA_BF16, M, 2 * F, 2 * F), e = mk(io->e_q, CODA_E4M3, M, 2 * F, 2 * F);
    coda_epilogue_program pg = prog_of({CODA_OP_TENSOR_SCALE, CODA_OP_SWIGLU_BWD, CODA_OP_ROW_SCALE,
                                        CODA_OP_ROW_DOT_PARTIAL, CODA_OP_AMAX});
    coda_side_inputs sd{};
    sd.tensor_scale = io->s_dy * io->s_wd;
    sd.row_scale = io->r;
    sd.aux_in = &Z;
    sd.out_scale = 1.0f / io->s_e;
    coda_aux_outputs ax{};
    ax.row_partials = spart;
    ax.row_partials_ld = M;
    ax.amax = io->amax_e;
    if ((st = coda_gemm_epilogue(&dYq, &W, &pg, &sd, &e, &ax, stream)) != CODA_OK) return st;
  }
  if ((st = coda_rms_partial_reduce(spart, M, (int32_t)((F + 255) / 256), M, H, 0.f, CODA_REDUCE_SCALE_SUM, io->r,
                                    io->c, stream)) != CODA_OK)
    return st;
  {
    // dW_d = s_dy s_a (dY_q^T a_q)
    coda_tensor A = mk(io->dY_q, CODA_E4M3, H, M, H, CODA_COL_MAJOR);
    coda_tensor W = mk(io->a_q, CODA_E4M3, F, M, F, CODA_COL_MAJOR);
    coda_tensor out = mk(io->dW_d, CODA_F32, H, F, F);
    coda_epilogue_program pg = prog_of({CODA_OP_TENSOR_SCALE});
    coda_side_inputs sd{};
    sd.tensor_scale = io->s_dy * io->s_a;
    if ((st = gemm_epilogue_impl(&A, &W, &pg, &sd, &out, nullptr, stream, true)) != CODA_OK) return st;
  }
  {
    // dh = s_e s_w (e_q W_q) - c h + dY
    coda_tensor A = mk(io->e_q, CODA_E4M3, M, 2 * F, 2 * F);
    coda_tensor W = mk(io->W_q, CODA_E4M3, H, 2 * F, H, CODA_COL_MAJOR);   // logical W^T
    coda_tensor h = mk(io->h, CODA_BF16, M, H, H), out = mk(io->dh, CODA_BF16, M, H, H);
    coda_epilogue_program pg = prog_of({CODA_OP_TENSOR_SCALE, CODA_OP_RMSBWD_COMBINE});
    coda_side_inputs sd{};
    sd.tensor_scale = io->s_e * io->s_w;
    sd.row_coef = io->c;
    sd.aux_in = &h;
    sd.aux_in2 = &dY;
    if ((st = gemm_epilogue_impl(&A, &W, &pg, &sd, &out, nullptr, stream, true)) != CODA_OK) return st;
  }
  {
    // dW = s_e s_x (e_q^T X_q)
    coda_tensor A = mk(io->e_q, CODA_E4M3, 2 * F, M, 2 * F, CODA_COL_MAJOR);
    coda_tensor W = mk(io->X_q, CODA_E4M3, H, M, H, CODA_COL_MAJOR);
    coda_tensor out = mk(io->dW, CODA_F32, 2 * F, H, H);
    coda_epilogue_program pg = prog_of({CODA_OP_TENSOR_SCALE});
    coda_side_inputs sd{};
    sd.tensor_scale = io->s_e * io->s_x;
    if ((st = gemm_epilogue_impl(&A, &W, &pg, &sd, &out, nullptr, stream, true)) != CODA_OK) return st;
  }
  return CODA_OK;
}

int coda_mlp_nvfp4_backward(const coda_mlp_nvfp4_bwd_io* io, void* stream) {
  if (!io) return CODA_ERR_NULL;
  const int64_t M = io->M, H = io->H, F = io->F;
  if (M < 0 || M % 256 != 0 || H < 256 || F < 256 || H % 256 != 0 || F % 256 != 0) return CODA_ERR_SHAPE;
  const float scales[6] = {io->s_x, io->s_wt, io->s_wdt, io->s_a, io->s_dy, io->s_e};
  for (float v : scales)
    if (!(v > 0.f) || !(v < INFINITY)) return CODA_ERR_SHAPE;
  if (!io->W_guT || !io->W_guT_sf || !io->W_dT || !io->W_dT_sf || !io->amax_dy || !io->amax_e || !io->dW_d || !io->dW)
    return CODA_ERR_NULL;
  if (M > 0 && (!io->h || !io->Z || !io->r || !io->dY || !io->dY_r || !io->dY_r_sf || !io->dY_c || !io->dY_c_sf ||
                !io->e || !io->e_r || !io->e_r_sf || !io->e_c || !io->e_c_sf || !io->a_c || !io->a_c_sf ||
                !io->x_c || !io->x_c_sf || !io->c || !io->dh || !io->workspace))
    return CODA_ERR_NULL;
  if (M > 0 && !aligned16(io->workspace)) return CODA_ERR_ALIGN;
  int st;
  DevState* dv;
  if ((st = ensure_device(&dv)) != CODA_OK) return st;
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(io->amax_dy, 0, sizeof(float), cs) != cudaSuccess ||
      cudaMemsetAsync(io->amax_e, 0, sizeof(float), cs) != cudaSuccess)
    return CODA_ERR_LAUNCH;
  if (M == 0) {   // sums over an empty batch: zero weight gradients
    if (cudaMemsetAsync(io->dW_d, 0, (size_t)H * F * sizeof(float), cs) != cudaSuccess ||
        cudaMemsetAsync(io->dW, 0, (size_t)2 * F * H * sizeof(float), cs) != cudaSuccess)
      return CODA_ERR_LAUNCH;
    return CODA_OK;
  }
  // dY along its rows (for dA, K = H) and along its columns (for dW_d, K = tokens)
  coda_tensor dY = mk(io->dY, CODA_BF16, M, H, H);
  coda_tensor dYr = mk(io->dY_r, CODA_NVFP4, M, H, H), dYc = mk(io->dY_c, CODA_NVFP4, H, M, M);
  if ((st = coda_quantize_nvfp4_t(&dY, CODA_QT_PLAIN, io->s_dy, &dYc, io->dY_c_sf, &dYr, io->dY_r_sf, io->amax_dy,
                                   stream)) != CODA_OK)
    return st;
  float* spart = io->workspace;   // [ceil(F / 128), M] row partials of sum e . Z (one per 128-column tile)
  coda_tensor e = mk(io->e, CODA_BF16, M, 2 * F, 2 * F);
  coda_tensor Z = mk(io->Z, CODA_BF16, M, 2 * F, 2 * F);
  {
    // dA = s_dy s_wdt (dY_r W_dT^T); SwiGLU backward with r; e in bf16, row partials of e . Z
    coda_tensor W = mk(io->W_dT, CODA_NVFP4, F, H, H);
    coda_epilogue_program pg = prog_of({CODA_OP_TENSOR_SCALE, CODA_OP_SWIGLU_BWD, CODA_OP_ROW_SCALE,
                                        CODA_OP_ROW_DOT_PARTIAL});
    coda_side_inputs sd{};
    sd.tensor_scale = io->s_dy * io->s_wdt;
    sd.row_scale = io->r;
    sd.aux_in = &Z;
    sd.a_block_scales = io->dY_r_sf;
    sd.w_block_scales = io->W_dT_sf;
    coda_aux_outputs ax{};
    ax.row_partials = spart;
    ax.row_partials_ld = M;
    if ((st = gemm_epilogue_impl(&dYr, &W, &pg, &sd, &e, &ax, stream, true)) != CODA_OK) return st;
  }
  if ((st = coda_rms_partial_reduce(spart, M, (int32_t)((F + 127) / 128), M, H, 0.f, CODA_REDUCE_SCALE_SUM, io->r,
                                    io->c, stream)) != CODA_OK)
    return st;
  // e along its rows (for t = e W_gu, K = 2F) and along its columns (for dW, K = tokens); a
  // from the saved Z and h, along their columns (for dW_d and dW)
  coda_tensor er = mk(io->e_r, CODA_NVFP4, M, 2 * F, 2 * F), ec = mk(io->e_c, CODA_NVFP4, 2 * F, M, M);
  coda_tensor ac = mk(io->a_c, CODA_NVFP4, F, M, M), xc = mk(io->x_c, CODA_NVFP4, H, M, M);
  coda_tensor h = mk(io->h, CODA_BF16, M, H, H);
  if ((st = coda_quantize_nvfp4_t(&e, CODA_QT_PLAIN, io->s_e, &ec, io->e_c_sf, &er, io->e_r_sf, io->amax_e,
                                   stream)) != CODA_OK)
    return st;
  if ((st = coda_quantize_nvfp4_t(&Z, CODA_QT_SWIGLU, io->s_a, &ac, io->a_c_sf, nullptr, nullptr, nullptr, stream)) !=
      CODA_OK)
    return st;
  if ((st = coda_quantize_nvfp4_t(&h, CODA_QT_PLAIN, io->s_x, &xc, io->x_c_sf, nullptr, nullptr, nullptr, stream)) !=
      CODA_OK)
    return st;
  {
    // dW_d = s_dy s_a (dY_c a_c^T), contracting over the tokens
    coda_tensor out = mk(io->dW_d, CODA_F32, H, F, F);
    coda_epilogue_program pg = prog_of({CODA_OP_TENSOR_SCALE});
    coda_side_inputs sd{};
    sd.tensor_scale = io->s_dy * io->s_a;
    sd.a_block_scales = io->dY_c_sf;
    sd.w_block_scales = io->a_c_sf;
    if ((st = gemm_epilogue_impl(&dYc, &ac, &pg, &sd, &out, nullptr, stream, true)) != CODA_OK) return st;
  }
  {
    // dh = s_e s_wt (e_r W_guT^T) - c h + dY
    coda_tensor W = mk(io->W_guT, CODA_NVFP4, H, 2 * F, 2 * F), out = mk(io->dh, CODA_BF16, M, H, H);
    coda_epilogue_program pg = prog_of({CODA_OP_TENSOR_SCALE, CODA_OP_RMSBWD_COMBINE});
    coda_side_inputs sd{};
    sd.tensor_scale = io->s_e * io->s_wt;
    sd.row_coef = io->c;
    sd.aux_in = &h;
    sd.aux_in2 = &dY;
    sd.a_block_scales = io->e_r_sf;
    sd.w_block_scales = io->W_guT_sf;
    if ((st = gemm_epilogue_impl(&er, &W, &pg, &sd, &out, nullptr, stream, true)) != CODA_OK) return st;
  }
  {
    // dW = s_e s_x (e_c x_c^T), contracting over the tokens
    coda_tensor out = mk(io->dW, CODA_F32, 2 * F, H, H);
    coda_epilogue_program pg = prog_of({CODA_OP_TENSOR_SCALE});
    coda_side_inputs sd{};
    sd.tensor_scale = io->s_e * io->s_x;
    sd.a_block_scales = io->e_c_sf;
    sd.w_block_scales = io->x_c_sf;
    if ((st = gemm_epilogue_impl(&ec, &xc, &pg, &sd, &out, nullptr, stream, true)) != CODA_OK) return st;
  }
  return CODA_OK;
}

}  // extern "C"
