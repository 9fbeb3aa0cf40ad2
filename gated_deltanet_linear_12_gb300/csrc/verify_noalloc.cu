// gdn_verify_step_noalloc: the read-only verify with its workspace in a fixed
// device buffer owned by the library, for callers that cannot allocate device
// memory themselves (see include/gdn.h).
//
// The buffer is a file-scope device array. Host code cannot use the array's
// name as a device address (on the host it names a stand-in object), so the
// real address is looked up with cudaGetSymbolAddress once per device, with
// that device current, and handed to the kernels as their workspace pointer.
// Nothing here allocates: no cudaMalloc, no cudaFree, no allocating library call.
#include <cuda_runtime.h>

#include <mutex>

#include "gdn.h"

namespace {

static __device__ __align__(256) uint8_t g_verify_scratch[GDN_VERIFY_NOALLOC_MAX_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device; looked up on the
// first call made with that device current.
gdn_status scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_verify_step_noalloc(const gdn_config* cfg, const void* x, const void* conv_w,
                                              const void* conv_state, const float* state, const float* alpha,
                                              const float* beta, const void* z, const float* norm_w, void* out,
                                              const int32_t* slot_idx, int32_t B, int32_t T, void* postconv_out,
                                              void* stream) {
  const int64_t need = gdn_verify_workspace_bytes(cfg, B, T);
  if (need < 0) return GDN_ERR_INVALID;
  if (need > (int64_t)GDN_VERIFY_NOALLOC_MAX_BYTES) return GDN_ERR_UNSUPPORTED;
  if (B == 0) return GDN_OK;
  void* scratch = nullptr;
  const gdn_status st = scratch_on_current_device(&scratch);
  if (st != GDN_OK) return st;
  // The read-only verify never writes conv_state or state.
  return gdn_verify_step(cfg, x, conv_w, const_cast<void*>(conv_state), const_cast<float*>(state), alpha, beta, z,
                         norm_w, out, slot_idx, B, T, 0u, postconv_out, scratch, GDN_VERIFY_NOALLOC_MAX_BYTES,
                         stream);
}
