// coda_block_forward_noalloc: the block forward chain for callers that cannot allocate
// device memory.  The chain's only scratch — the per-tile partial sums of squares that G1
// writes and the row reduce reads — lives in a fixed-size array in this file instead of a
// caller-provided workspace.  Everything else is the existing coda_block_forward.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/coda.h"

// The static scratch: CODA_NOALLOC_MAX_PARTIALS floats (4 MiB), held by every device that
// loads the library until the process exits.
static __device__ __align__(256) float g_noalloc_partials[CODA_NOALLOC_MAX_PARTIALS];

namespace {

constexpr int kMaxDevices = 64;
float* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the scratch on the current device.  In host code the array's name is
// only a host-side stand-in, so the address is looked up once per device, with that device
// current, and cached.
int scratch_on_current_device(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return CODA_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_partials) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return CODA_ERR_NO_DEVICE;
    }
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
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
