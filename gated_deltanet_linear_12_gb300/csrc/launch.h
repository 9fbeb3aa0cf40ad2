// Internal launcher interface between the C ABI (gdn_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "gdn.h"

namespace gdn {

// Kernel attributes (the dynamic shared memory limit, optionally the largest
// shared-memory carveout), set once per kernel and device, and again only when a
// launch needs a larger limit than any before: each call costs host time that a
// small launch cannot hide.
template <auto Kern>
cudaError_t set_smem_once(int smem_bytes, bool max_carveout = false) {
  static std::atomic<int> limit[64];                     // per device: the limit set so far
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool cached = dev >= 0 && dev < 64;
  if (cached && limit[dev].load(std::memory_order_acquire) >= smem_bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e == cudaSuccess && max_carveout)
    e = cudaFuncSetAttribute(Kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess && cached) {
    int cur = limit[dev].load(std::memory_order_relaxed);
    while (cur < smem_bytes && !limit[dev].compare_exchange_weak(cur, smem_bytes, std::memory_order_acq_rel)) {
    }
  }
  return e;
}

// Number of SMs of the current device, looked up once per device.
inline cudaError_t sm_count(int* n) {
  static std::atomic<int> cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) { *n = c; return cudaSuccess; }
  }
  e = cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess && dev >= 0 && dev < 64) cache[dev].store(*n, std::memory_order_relaxed);
  return e;
}

struct StepArgs {
  const void* x;            // [B][T][C]
  const void* conv_w;       // [C][4]
  void* conv_state;         // pool
  float* state;             // pool
  const void* alpha;        // [B][T][Hv] gate dtype
  const void* beta;
  const void* z;            // [B][T][Hv*D]
  const float* norm_w;      // [D]
  void* out;                // [B][T][Hv*D]
  void* postconv;           // nullable [B][T][C]
  const int32_t* slot_idx;  // [B]
  const int32_t* n_keep;    // [B] (commit)
  const gdn_layer_view* layers;  // [L] (commit)
  int B, T, Hk, Hv, n_slots;
  float eps, q_scale;
  uint32_t* dev_err;
  int raw_gates;            // alpha / beta hold raw projections: apply the gate step
  int gate_bf16;            // gate arrays hold bf16 values
  int out_f32;              // out is f32 (else the activation dtype)
  // verify with the previous window's commit folded in (n_keep: its accepted prefixes)
  const void* prev_x;       // [B][prev_T][C]
  const void* prev_alpha;   // [B][prev_T][Hv]
  const void* prev_beta;
  int prev_T;
};

struct PrefillArgs {
  const void* qkv;
  const void* alpha;        // [n_tok][Hv] gate dtype
  const void* beta;
  const void* z;
  const float* norm_w;
  void* out;
  float* state;
  const int32_t* slot_idx;
  const int32_t* cu;
  const uint8_t* has_init;
  int n_seq, Hk, Hv, n_slots;
  int64_t n_tok;
  float eps, q_scale;
  uint32_t* dev_err;
  int raw_gates;            // alpha / beta hold raw projections: apply the gate step
  int gate_bf16;            // gate arrays hold bf16 values
  int out_f32;              // out is f32 (else the activation dtype)
};

// Encodes a 2-D row-major bf16 tensor map (rows x cols, row pitch in elements)
// copied in boxes of box_cols x box_rows, without swizzle; out-of-range rows
// read as zeros.
cudaError_t encode_bf16_rows_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                                 uint64_t pitch, uint32_t box_cols, uint32_t box_rows);
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();

cudaError_t launch_conv_fwd(const gdn_config& cfg, const void* x, int64_t ld_x, void* y,
                            int64_t ld_y, const void* conv_w, void* conv_state,
                            const int32_t* slot_idx, const int32_t* cu, const uint8_t* has_init,
                            int n_seq, int64_t n_tok, int fuse_norm, cudaStream_t stream);
cudaError_t launch_postconv_norm(const gdn_config& cfg, int in_t, const void* yin, int out_t,
                                 void* yout, int64_t n_tok, int n_sm, cudaStream_t stream);
cudaError_t launch_verify(const StepArgs& a, bool commit_all, int act, cudaStream_t stream);
cudaError_t launch_verify_readonly(const StepArgs& a, int act, cudaStream_t stream);
cudaError_t launch_commit(const StepArgs& a, int L, int act, cudaStream_t stream);
cudaError_t launch_verify_lazy(const StepArgs& a, int act, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillArgs& a, int act, cudaStream_t stream);
cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_gates(const void* a, const void* b, void* alpha, void* beta, int64_t n, int bf16,
                         cudaStream_t stream);

}  // namespace gdn
