// gdn_verify_step_noalloc: the read-only verify for callers that cannot
// allocate device memory themselves (see include/gdn.h). The verify kernel keeps
// everything it computes in shared memory, registers and TMEM, so this entry
// point needs no buffer of its own: it validates its arguments like
// gdn_verify_step and launches the same kernel. Nothing here allocates: no
// cudaMalloc, no cudaFree, no allocating library call.
#include <cuda_runtime.h>

#include "gdn.h"

extern "C" gdn_status gdn_verify_step_noalloc(const gdn_config* cfg, const void* x, const void* conv_w,
                                              const void* conv_state, const float* state, const void* alpha,
                                              const void* beta, const void* z, const float* norm_w, void* out,
                                              const int32_t* slot_idx, int32_t B, int32_t T, void* postconv_out,
                                              void* stream) {
  // The read-only verify never writes conv_state or state.
  return gdn_verify_step(cfg, x, conv_w, const_cast<void*>(conv_state), const_cast<float*>(state), alpha, beta, z,
                         norm_w, out, slot_idx, B, T, 0u, postconv_out, nullptr, 0, stream);
}
