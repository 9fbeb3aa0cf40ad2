// The gate step as its own launch: alpha = exp(-softplus(a)), beta = sigmoid(b)
// over n values ("Strata PR #3226" tests a fused gate kernel against its
// multi-token form; the formula is the synthetic workloads' form of the gates).
// Elementwise and HBM-bound: 16 bytes read and 8 written per value, four values
// per thread as 16-byte loads and stores, a grid-stride loop over a grid of
// a few blocks per SM. gate_alpha / gate_beta are the device functions the
// prefill, verify and commit kernels apply in GDN_GATES_RAW mode, so both
// routes give the same bits.
#include "common.cuh"
#include "launch.h"

namespace gdn {

namespace {

__global__ void __launch_bounds__(256) gates_kernel(const float* a, const float* b,
                                                    float* alpha, float* beta, int64_t n) {
  const int64_t n4 = n >> 2;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const bool vec = ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) |
                     reinterpret_cast<uintptr_t>(alpha) | reinterpret_cast<uintptr_t>(beta)) & 15u) == 0;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (vec) {
    for (int64_t q = i; q < n4; q += stride) {
      const float4 av = reinterpret_cast<const float4*>(a)[q];
      const float4 bv = reinterpret_cast<const float4*>(b)[q];
      reinterpret_cast<float4*>(alpha)[q] =
          make_float4(gate_alpha(av.x), gate_alpha(av.y), gate_alpha(av.z), gate_alpha(av.w));
      reinterpret_cast<float4*>(beta)[q] =
          make_float4(gate_beta(bv.x), gate_beta(bv.y), gate_beta(bv.z), gate_beta(bv.w));
    }
    i += n4 * 4;                                         // the tail, one value per thread
  }
  for (; i < n; i += stride) {
    const float av = a[i], bv = b[i];
    alpha[i] = gate_alpha(av);
    beta[i] = gate_beta(bv);
  }
}

}  // namespace

cudaError_t launch_gates(const float* a, const float* b, float* alpha, float* beta, int64_t n,
                         cudaStream_t stream) {
  int n_sm = 0;
  cudaError_t e = sm_count(&n_sm);
  if (e != cudaSuccess) return e;
  const int64_t want = (n / 4 + 255) / 256;
  const int64_t cap = (int64_t)n_sm * 8;
  const unsigned grid = (unsigned)(want < 1 ? 1 : want > cap ? cap : want);
  gates_kernel<<<grid, 256, 0, stream>>>(a, b, alpha, beta, n);
  return cudaGetLastError();
}

}  // namespace gdn
