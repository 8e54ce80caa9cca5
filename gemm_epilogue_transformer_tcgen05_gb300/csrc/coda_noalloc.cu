// coda_block_forward_noalloc: the block forward chain for callers that cannot allocate
// device memory.  The chain's only scratch — the per-tile partial sums of squares that G1
// writes and the row reduce reads — lives in a fixed-size array in this file instead of a
// caller-provided workspace.  Everything else is the existing coda_block_forward.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/coda.h"

// The static scratch: CODA_NOALLOC_MAX_PARTIALS floats (4 MiB), held by every device that
// loads the library until the process exits.
static __device__ __align__(256) float g_noalloc_partials[CODA_NOALLOC_MAX_PARTIALS];

namespace {

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  float* ptr = nullptr;
  unsigned long long ctx_id = 0;  // the context the address belongs to
};
ScratchSlot g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

typedef CUresult (*PfnCtxGetCurrent)(CUcontext*);
typedef CUresult (*PfnCtxGetId)(CUcontext, unsigned long long*);
PfnCtxGetCurrent g_ctx_get_current = nullptr;
PfnCtxGetId g_ctx_get_id = nullptr;
bool g_ctx_fns_looked_up = false;

// Unique id of the current context (0 when it cannot be read).  A device reset destroys the
// context and the next runtime call creates a new one with a new id, where the array may sit
// at another address.
unsigned long long current_context_id() {
  if (!g_ctx_fns_looked_up) {
    g_ctx_fns_looked_up = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_current = reinterpret_cast<PfnCtxGetCurrent>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_id = reinterpret_cast<PfnCtxGetId>(fn);
    cudaGetLastError();
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_get_current && g_ctx_get_id && g_ctx_get_current(&ctx) == CUDA_SUCCESS && ctx &&
      g_ctx_get_id(ctx, &id) == CUDA_SUCCESS)
    return id;
  return 0;
}

// Device address of the scratch on the current device.  In host code the array's name is
// only a host-side stand-in, so the address is looked up with the device current, on the
// first call in each context, and cached for that context.
int scratch_on_current_device(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return CODA_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  const unsigned long long ctx = current_context_id();
  ScratchSlot& slot = g_scratch[dev];
  if (!slot.ptr || ctx == 0 || slot.ctx_id != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_partials) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return CODA_ERR_NO_DEVICE;
    }
    slot.ptr = static_cast<float*>(p);
    slot.ctx_id = current_context_id();  // the look-up made the device's context current
  }
  *out = slot.ptr;
  return CODA_OK;
}

}  // namespace

extern "C" int coda_block_forward_noalloc(const coda_block_fwd* io, void* stream) {
  if (!io) return CODA_ERR_NULL;
  if (io->workspace != nullptr) return CODA_ERR_SHAPE;  // the scratch is internal here
  if (io->M < 0 || io->H < 1) return CODA_ERR_SHAPE;
  const int64_t nparts = (io->H + 255) / 256;
  if (io->M > 0 && nparts > (int64_t)CODA_NOALLOC_MAX_PARTIALS / io->M) return CODA_ERR_SHAPE;
  float* scratch = nullptr;
  const int st = scratch_on_current_device(&scratch);
  if (st != CODA_OK) return st;
  coda_block_fwd local = *io;
  local.workspace = scratch;
  return coda_block_forward(&local, stream);
}
