// Shared device helpers of the GDN kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr int D = 128;        // head_dim
constexpr int KW = 4;         // conv width
constexpr int KS = KW - 1;    // conv_state rows
constexpr int CHUNK = 64;     // exact chunk of the conv and of the prefill
constexpr int MAXT = 8;       // draft tokens of a verify window
constexpr unsigned FULL = 0xffffffffu;

enum Act { F32 = 0, BF16 = 1 };

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }
__device__ __forceinline__ uint16_t f2bf(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Value after a store in activation type A (round to bf16 or keep f32).
template <int A> __device__ __forceinline__ float round_act(float f) {
  if constexpr (A == BF16) return bf2f(f2bf(f));
  else return f;
}

// Load / store 8 contiguous activations starting at element `i` of `base`.
// bf16: one 16-byte access; f32: two.
template <int A> __device__ __forceinline__ void load8(const void* base, int64_t i, float v[8]) {
  if constexpr (A == BF16) {
    uint4 u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + i);
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = __uint_as_float(w[j] << 16);
      v[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + i);
    float4 a = p[0], b = p[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

template <int A> __device__ __forceinline__ void store8(void* base, int64_t i, const float v[8]) {
  if constexpr (A == BF16) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
      w[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + i) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + i);
    p[0] = make_float4(v[0], v[1], v[2], v[3]);
    p[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

// Eight activations kept packed between load and use (4 registers for bf16).
template <int A> struct Raw8;
template <> struct Raw8<BF16> { uint4 u; };
template <> struct Raw8<F32> { float4 a, b; };

template <int A> __device__ __forceinline__ void raw_load(const void* base, int64_t i, Raw8<A>& r) {
  if constexpr (A == BF16) r.u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + i);
  else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + i);
    r.a = p[0];
    r.b = p[1];
  }
}
template <int A> __device__ __forceinline__ void raw_zero(Raw8<A>& r) {
  if constexpr (A == BF16) r.u = make_uint4(0u, 0u, 0u, 0u);
  else { r.a = make_float4(0.f, 0.f, 0.f, 0.f); r.b = r.a; }
}
template <int A> __device__ __forceinline__ void raw_unpack(const Raw8<A>& r, float v[8]) {
  if constexpr (A == BF16) {
    const uint32_t w[4] = {r.u.x, r.u.y, r.u.z, r.u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[2 * j] = __uint_as_float(w[j] << 16);
      v[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  } else {
    v[0] = r.a.x; v[1] = r.a.y; v[2] = r.a.z; v[3] = r.a.w;
    v[4] = r.b.x; v[5] = r.b.y; v[6] = r.b.z; v[7] = r.b.w;
  }
}

// Output rows: the activation dtype A, or f32 when out_f32.
template <int A> __device__ __forceinline__ void store_out8(void* base, int64_t i, const float v[8], int out_f32) {
  if (out_f32) store8<F32>(base, i, v);
  else store8<A>(base, i, v);
}

// One gate value (alpha, beta or a raw projection) widened to f32.
__device__ __forceinline__ float load_gate(const void* p, int64_t i, int bf16) {
  return bf16 ? bf2f(static_cast<const uint16_t*>(p)[i]) : static_cast<const float*>(p)[i];
}

__device__ __forceinline__ void report(uint32_t* dev_err, uint32_t bit) {
  if (dev_err) atomicOr(dev_err, bit);
}

// Causal conv of one channel: the tap products summed from zero in tap order,
// tap 3 on the current token, each product and each sum rounded on its own.
// Scalar __fmul_rn / __fadd_rn are never merged into fused multiply-adds.
__device__ __forceinline__ float conv4(const float w[4], float x0, float x1, float x2, float x3) {
  float acc = __fmul_rn(w[0], x0);
  acc = __fadd_rn(acc, __fmul_rn(w[1], x1));
  acc = __fadd_rn(acc, __fmul_rn(w[2], x2));
  acc = __fadd_rn(acc, __fmul_rn(w[3], x3));
  return acc;
}

// The same for two channels at once (w0..w3 hold the taps of both). With bf16
// operands every product is exact in f32 (8 x 8 significant bits), so a fused
// multiply-add rounds exactly like a rounded product followed by a rounded
// sum: the paired fused form gives the bits of conv4. f32 operands take conv4.
template <int A>
__device__ __forceinline__ float2 conv4x2(float2 w0, float2 w1, float2 w2, float2 w3, float2 x0,
                                          float2 x1, float2 x2, float2 x3) {
  if constexpr (A == BF16) {
    float2 acc = __fmul2_rn(w0, x0);
    acc = __ffma2_rn(w1, x1, acc);
    acc = __ffma2_rn(w2, x2, acc);
    acc = __ffma2_rn(w3, x3, acc);
    return acc;
  } else {
    const float wa[4] = {w0.x, w1.x, w2.x, w3.x}, wb[4] = {w0.y, w1.y, w2.y, w3.y};
    return make_float2(conv4(wa, x0.x, x1.x, x2.x, x3.x), conv4(wb, x0.y, x1.y, x2.y, x3.y));
  }
}

// SiLU y / (1 + e^-y), computed as y * 1 / (1 + 2^(-y log2 e)) with the
// hardware power of two and reciprocal approximations (ftz) written out: one
// multiply, two MUFU operations, one add and one multiply. Relative error
// against the exact value: a few ulp plus |y| 2^-24 from the rounding of the
// exponent's argument (below 2e-6 for |y| <= 30); for y < -88 the power
// overflows and the result is -0, against an exact value below 6e-37 in
// magnitude.
__device__ __forceinline__ float hw_ex2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float hw_rcp(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float silu(float y) {
  constexpr float kNegLog2e = -1.4426950408889634f;     // -1 / ln 2
  return __fmul_rn(y, hw_rcp(__fadd_rn(1.0f, hw_ex2(__fmul_rn(y, kNegLog2e)))));
}
__device__ __forceinline__ float2 silu2(float2 y) { return make_float2(silu(y.x), silu(y.y)); }

// SiLU of the output gate z: the same function.
__device__ __forceinline__ float silu_gate(float z) { return silu(z); }

// The gate step from raw projections ("Strata PR #3226" names a fused gate
// kernel; the form is the one of the synthetic workloads' gates):
//   alpha = exp(-softplus(a)), softplus(a) = log(1 + e^a), taken as
//           a + log(1 + e^-a) for a > 0 so that e^a is never formed there;
//   beta  = 1 / (1 + e^-b), taken as e^b / (1 + e^b) for b < 0 (the same value
//           in exact arithmetic) so that e^-b never overflows there.
// CUDA's accurate expf / log1pf and correctly rounded adds, multiplies and
// divide: every kernel that applies the step gets the same bits as gdn_gates.
__device__ __forceinline__ float gate_alpha(float a) {
  const float sp = a > 0.0f ? __fadd_rn(a, log1pf(expf(-a))) : log1pf(expf(a));
  return expf(-sp);
}
__device__ __forceinline__ float gate_beta(float b) {
  const float e = expf(-fabsf(b));                      // in [0, 1]
  const float s = __fdiv_rn(1.0f, __fadd_rn(1.0f, e));  // sigmoid(|b|)
  return b >= 0.0f ? s : __fmul_rn(e, s);
}

// Sum of squares of a 128-channel head held as 8 contiguous channels by each
// of 16 consecutive lanes (lane & 15 = channel group). In-lane: strides 4, 2, 1;
// across lanes: xor 8, 4, 2, 1, which gives every lane the same bits because
// float addition is commutative. Must be called by all 32 lanes of the warp.
// Scalar __fmul_rn / __fadd_rn: these are never merged into multiply-adds,
// so each square is rounded before it is summed (paired f32 multiplies have
// been seen fused into the following paired add).
__device__ __forceinline__ float head_sum_sq16(const float v[8]) {
  float e[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) e[j] = __fmul_rn(v[j], v[j]);
  const float p0 = __fadd_rn(e[0], e[4]), p1 = __fadd_rn(e[1], e[5]);
  const float p2 = __fadd_rn(e[2], e[6]), p3 = __fadd_rn(e[3], e[7]);
  float g = __fadd_rn(__fadd_rn(p0, p2), __fadd_rn(p1, p3));
#pragma unroll
  for (int m = 8; m >= 1; m >>= 1) g = __fadd_rn(g, __shfl_xor_sync(FULL, g, m));
  return g;
}

// In-lane part of head_sum_sq16: the sum of squares of one lane's 8 channels,
// strides 4, 2, 1.
__device__ __forceinline__ float lane_sum_sq8(const float v[8]) {
  float e[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) e[j] = __fmul_rn(v[j], v[j]);
  const float p0 = __fadd_rn(e[0], e[4]), p1 = __fadd_rn(e[1], e[5]);
  const float p2 = __fadd_rn(e[2], e[6]), p3 = __fadd_rn(e[3], e[7]);
  return __fadd_rn(__fadd_rn(p0, p2), __fadd_rn(p1, p3));
}

// The 1 / sqrt(ss + eps) of eight tokens u = 0..7 of a 128-channel head whose
// in-lane sums g[u] (lane_sum_sq8) 16 consecutive lanes hold, with the bits of
// head_sum_sq16 + inv_norm per token. Across lanes the eight sums are reduced by
// halving exchanges: at xor 8 a lane keeps four tokens (its own half) and adds
// the partner's partial sums of them, then two at xor 4, one at xor 2, and xor 1
// pairs the two lanes that hold the same token. Every addition has
// head_sum_sq16's operands, so the sums are bitwise equal; 8 shuffles and one
// root per lane instead of 32 and eight. Returns the factor of this lane's
// token, 4 b3 + 2 b2 + b1 (lane bits); token u's factor is at lane
// token_lane(u) of the 16. Must be called by all 32 lanes of the warp.
__device__ __forceinline__ float inv_norm(float ss, float eps);
__device__ __forceinline__ float lanes_inv_norm8(const float (&g)[8], float eps) {
  const int lane = threadIdx.x & 31;
  const bool b3 = (lane & 8) != 0, b2 = (lane & 4) != 0, b1 = (lane & 2) != 0;
  float h4[4], h2[2];
#pragma unroll
  for (int k = 0; k < 4; ++k) {                       // tokens 4 b3 + k
    const float send = b3 ? g[k] : g[k + 4], keep = b3 ? g[k + 4] : g[k];
    h4[k] = __fadd_rn(keep, __shfl_xor_sync(FULL, send, 8));
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {                       // tokens 4 b3 + 2 b2 + k
    const float send = b2 ? h4[k] : h4[k + 2], keep = b2 ? h4[k + 2] : h4[k];
    h2[k] = __fadd_rn(keep, __shfl_xor_sync(FULL, send, 4));
  }
  const float send = b1 ? h2[0] : h2[1], keep = b1 ? h2[1] : h2[0];
  const float h1 = __fadd_rn(keep, __shfl_xor_sync(FULL, send, 2));
  return inv_norm(__fadd_rn(h1, __shfl_xor_sync(FULL, h1, 1)), eps);
}
__host__ __device__ constexpr int token_lane(int u) { return ((u >> 2) << 3) | (((u >> 1) & 1) << 2) | ((u & 1) << 1); }

// 1 / sqrt(ss + eps) with correctly rounded root and divide.
__device__ __forceinline__ float inv_norm(float ss, float eps) {
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ss, eps)));
}

// Chunk lookup for exact per-sequence chunks: chunk j (global) -> sequence s
// and chunk ci inside it, every sequence owning max(1, ceil(len / chunk))
// chunks. Executed by a whole warp; returns false if j is past the last chunk.
__device__ __forceinline__ bool find_chunk(const int32_t* __restrict__ cu, int n_seq, int j,
                                           int chunk, int& s_out, int& ci_out) {
  const int lane = threadIdx.x & 31;
  int base = 0;
  for (int s0 = 0; s0 < n_seq; s0 += 32) {
    const int s = s0 + lane;
    int cnt = 0;
    if (s < n_seq) {
      const int len = cu[s + 1] - cu[s];
      cnt = len > 0 ? (len + chunk - 1) / chunk : 1;
    }
    int inc = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(FULL, inc, o);
      if (lane >= o) inc += v;
    }
    const int exc = inc - cnt;
    const unsigned hit = __ballot_sync(FULL, s < n_seq && j >= base + exc && j < base + inc);
    if (hit) {
      const int l = __ffs(hit) - 1;
      s_out = s0 + l;
      ci_out = j - base - __shfl_sync(FULL, exc, l);
      return true;
    }
    base += __shfl_sync(FULL, inc, 31);
  }
  return false;
}

}  // namespace gdn
