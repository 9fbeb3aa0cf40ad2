// Self-test of the tensor-core building block: one block computes
// D[128][N] = A[128][K] * B[N][K]^T with tcgen05.mma (bf16 -> f32 in TMEM).
#include "common.cuh"
#include "gdn_selftest.h"
#include "tc.cuh"

namespace gdn {

// Operands only: A 128 x K and B N x K bf16, at most 32 KB + 64 KB. Every
// descriptor read ends inside its tile: A at 128 K 2 bytes, B at N K 2 bytes.
inline int tc_st_smem(int N, int K) { return (128 + N) * K * 2; }

__global__ void __launch_bounds__(128, 1)
tc_selftest_kernel(const uint16_t* __restrict__ A, const uint16_t* __restrict__ B,
                   float* __restrict__ Dout, int N, int K, int starve, uint32_t* err) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ uint64_t mbar;
  __shared__ uint32_t tslot;
  uint8_t* As = sm;
  uint8_t* Bs = sm + 128 * K * 2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kb_n = K / 8;
  for (int e = tid; e < 128 * kb_n; e += 128) {
    const int m = e / kb_n, kb = e % kb_n;
    *reinterpret_cast<uint4*>(As + tc::kmajor_offset(m, 8 * kb, 128)) =
        *reinterpret_cast<const uint4*>(A + (size_t)m * K + 8 * kb);
  }
  for (int e = tid; e < N * kb_n; e += 128) {
    const int n = e / kb_n, kb = e % kb_n;
    *reinterpret_cast<uint4*>(Bs + tc::kmajor_offset(n, 8 * kb, N)) =
        *reinterpret_cast<const uint4*>(B + (size_t)n * K + 8 * kb);
  }
  if (tid == 0) tc::mbar_init(&mbar, 1);
  tc::fence_async_smem();
  __syncthreads();
  uint32_t ncols = 32;
  while ((int)ncols < N) ncols <<= 1;
  if (warp == 0) {
    tc::tmem_alloc(&tslot, ncols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = tslot;
  if (tid == 0) {
    const uint32_t idesc = tc::idesc_bf16_f32(128, N);
    const uint32_t lboA = 16 * 128, sboA = 128;    // K neighbour, row neighbour
    const uint32_t lboB = (N / 8) * 128, sboB = 128;
    for (int ks = 0; ks < K / 16; ++ks) {
      const uint64_t ad = tc::smem_desc(tc::smem_u32(As) + ks * 2 * (16 * 128), lboA, sboA);
      const uint64_t bd = tc::smem_desc(tc::smem_u32(Bs) + ks * 2 * ((N / 8) * 128), lboB, sboB);
      tc::mma_bf16(tbase, ad, bd, idesc, ks > 0);
    }
    if (!starve) tc::mma_commit(&mbar);
  }
  // starve: nothing ever arrives on the barrier (the completion of the MMAs is
  // not attached to it), so the bounded wait must give up and report.
  const uint32_t polls = starve ? 4096u : (1u << 22);
  bool ok = tc::mbar_wait(&mbar, 0, polls);
  if (!ok) {
    if (err) atomicOr(err, 1u);
    if (starve) {                                   // attach the MMAs now, then drain them
      if (tid == 0) tc::mma_commit(&mbar);
      tc::mbar_wait(&mbar, 0, 1u << 22);
    } else {
      tc::mbar_wait(&mbar, 0, 1u << 22);            // give the MMAs in flight a second chance
    }
  }
  tc::fence_after_sync();
  if (ok) {
    for (int c = 0; c < N; c += 16) {
      float v[16];
      tc::tmem_ld16(tbase + ((uint32_t)(32 * warp) << 16) + c, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) Dout[(size_t)(32 * warp + lane) * N + c + i] = v[i];
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, ncols);
}

// The same product with f32 operands on the tf32 path (kind::tf32, K = 8 per
// instruction); A 128 x K and B N x K f32, at most 64 KB + 128 KB.
__global__ void __launch_bounds__(128, 1)
tc_selftest_tf32_kernel(const float* __restrict__ A, const float* __restrict__ B, float* __restrict__ Dout,
                        int N, int K, uint32_t* err) {
  extern __shared__ __align__(128) uint8_t sm[];
  __shared__ uint64_t mbar;
  __shared__ uint32_t tslot;
  uint8_t* As = sm;
  uint8_t* Bs = sm + 128 * K * 4;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kq = K / 4;
  for (int e = tid; e < 128 * kq; e += 128) {
    const int m = e / kq, kb = e % kq;
    *reinterpret_cast<float4*>(As + tc::kmajor32_offset(m, 4 * kb, 128)) =
        *reinterpret_cast<const float4*>(A + (size_t)m * K + 4 * kb);
  }
  for (int e = tid; e < N * kq; e += 128) {
    const int n = e / kq, kb = e % kq;
    *reinterpret_cast<float4*>(Bs + tc::kmajor32_offset(n, 4 * kb, N)) =
        *reinterpret_cast<const float4*>(B + (size_t)n * K + 4 * kb);
  }
  if (tid == 0) tc::mbar_init(&mbar, 1);
  tc::fence_async_smem();
  __syncthreads();
  uint32_t ncols = 32;
  while ((int)ncols < N) ncols <<= 1;
  if (warp == 0) {
    tc::tmem_alloc(&tslot, ncols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = tslot;
  if (tid == 0) {
    const uint32_t idesc = tc::idesc_tf32_f32(128, N);
    const uint32_t lboA = 16 * 128, sboA = 128;             // K neighbour, row neighbour
    const uint32_t lboB = (N / 8) * 128, sboB = 128;
    for (int ks = 0; ks < K / 8; ++ks) {
      const uint64_t ad = tc::smem_desc(tc::smem_u32(As) + ks * 2 * lboA, lboA, sboA);
      const uint64_t bd = tc::smem_desc(tc::smem_u32(Bs) + ks * 2 * lboB, lboB, sboB);
      tc::mma_tf32(tbase, ad, bd, idesc, ks > 0);
    }
    tc::mma_commit(&mbar);
  }
  const bool ok = tc::mbar_wait(&mbar, 0, 1u << 22);
  if (!ok) {
    if (err) atomicOr(err, 1u);
    tc::mbar_wait(&mbar, 0, 1u << 22);
  }
  tc::fence_after_sync();
  if (ok) {
    for (int c = 0; c < N; c += 16) {
      float v[16];
      tc::tmem_ld16(tbase + ((uint32_t)(32 * warp) << 16) + c, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) Dout[(size_t)(32 * warp + lane) * N + c + i] = v[i];
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, ncols);
}

}  // namespace gdn

extern "C" gdn_status gdn_selftest_tc_gemm_tf32(const float* A, const float* B, float* D, int32_t N,
                                                int32_t K, uint32_t* dev_err, void* stream) {
  if (!A || !B || !D) return GDN_ERR_INVALID;
  if (N < 16 || N > 256 || N % 16 || K < 8 || K > 128 || K % 8) return GDN_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) & 15u) return GDN_ERR_INVALID;
  const int smem = (128 + N) * K * 4;
  cudaError_t e = cudaFuncSetAttribute(gdn::tc_selftest_tf32_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return GDN_ERR_CUDA;
  gdn::tc_selftest_tf32_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(A, B, D, N, K, dev_err);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" gdn_status gdn_selftest_tc_gemm(const uint16_t* A, const uint16_t* B, float* D, int32_t N,
                                           int32_t K, int32_t starve_wait, uint32_t* dev_err,
                                           void* stream) {
  if (!A || !B || !D) return GDN_ERR_INVALID;
  if (N < 16 || N > 256 || N % 16 || K < 16 || K > 128 || K % 16) return GDN_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) & 15u) return GDN_ERR_INVALID;
  const int smem = gdn::tc_st_smem(N, K);
  cudaError_t e = cudaFuncSetAttribute(gdn::tc_selftest_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return GDN_ERR_CUDA;
  gdn::tc_selftest_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(
      A, B, D, N, K, starve_wait ? 1 : 0, dev_err);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
