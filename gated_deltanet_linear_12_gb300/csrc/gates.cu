// The gate step as its own launch: alpha = exp(-softplus(a)), beta = sigmoid(b)
// over n values ("Strata PR #3226" tests a fused gate kernel against its
// multi-token form; the formula is the synthetic workloads' form of the gates).
// Elementwise and HBM-bound: per value, a and b read, alpha and beta written
// (f32, four values per thread as 16-byte accesses; or bf16), a grid-stride loop
// over a grid of a few blocks per SM. gate_alpha / gate_beta are the device functions the
// prefill, verify and commit kernels apply in GDN_GATES_RAW mode, so both
// routes give the same bits.
#include "common.cuh"
#include "launch.h"

namespace gdn {

namespace {

template <bool BF> __device__ __forceinline__ float ld_g(const void* p, int64_t i) {
  if constexpr (BF) return bf2f(static_cast<const uint16_t*>(p)[i]);
  else return static_cast<const float*>(p)[i];
}
template <bool BF> __device__ __forceinline__ void st_g(void* p, int64_t i, float v) {
  if constexpr (BF) static_cast<uint16_t*>(p)[i] = f2bf(v);
  else static_cast<float*>(p)[i] = v;
}

// BF: a, b, alpha, beta hold bf16 values (read widened, results rounded to
// nearest even); else f32.
template <bool BF>
__global__ void __launch_bounds__(256) gates_kernel(const void* a, const void* b, void* alpha,
                                                    void* beta, int64_t n) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if constexpr (!BF) {
    const int64_t n4 = n >> 2;
    const bool vec = ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) |
                       reinterpret_cast<uintptr_t>(alpha) | reinterpret_cast<uintptr_t>(beta)) & 15u) == 0;
    if (vec) {
      for (int64_t q = i; q < n4; q += stride) {
        const float4 av = static_cast<const float4*>(a)[q];
        const float4 bv = static_cast<const float4*>(b)[q];
        static_cast<float4*>(alpha)[q] =
            make_float4(gate_alpha(av.x), gate_alpha(av.y), gate_alpha(av.z), gate_alpha(av.w));
        static_cast<float4*>(beta)[q] =
            make_float4(gate_beta(bv.x), gate_beta(bv.y), gate_beta(bv.z), gate_beta(bv.w));
      }
      i += n4 * 4;                                       // the tail, one value per thread
    }
  }
  for (; i < n; i += stride) {
    const float av = ld_g<BF>(a, i), bv = ld_g<BF>(b, i);
    st_g<BF>(alpha, i, gate_alpha(av));
    st_g<BF>(beta, i, gate_beta(bv));
  }
}

}  // namespace

cudaError_t launch_gates(const void* a, const void* b, void* alpha, void* beta, int64_t n, int bf16,
                         cudaStream_t stream) {
  int n_sm = 0;
  cudaError_t e = sm_count(&n_sm);
  if (e != cudaSuccess) return e;
  const int64_t want = (n / (bf16 ? 1 : 4) + 255) / 256;
  const int64_t cap = (int64_t)n_sm * 8;
  const unsigned grid = (unsigned)(want < 1 ? 1 : want > cap ? cap : want);
  if (bf16) gates_kernel<true><<<grid, 256, 0, stream>>>(a, b, alpha, beta, n);
  else gates_kernel<false><<<grid, 256, 0, stream>>>(a, b, alpha, beta, n);
  return cudaGetLastError();
}

}  // namespace gdn
