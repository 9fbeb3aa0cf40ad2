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

__device__ __forceinline__ void report(uint32_t* dev_err, uint32_t bit) {
  if (dev_err) atomicOr(dev_err, bit);
}

// Causal conv of one channel: taps in order, a rounded product then three
// fused multiply-adds, tap 3 on the current token.
__device__ __forceinline__ float conv4(const float w[4], float x0, float x1, float x2, float x3) {
  float acc = __fmul_rn(w[0], x0);
  acc = __fmaf_rn(w[1], x1, acc);
  acc = __fmaf_rn(w[2], x2, acc);
  acc = __fmaf_rn(w[3], x3, acc);
  return acc;
}

// The same for two channels at once (w0..w3 hold the taps of both).
__device__ __forceinline__ float2 conv4x2(float2 w0, float2 w1, float2 w2, float2 w3, float2 x0,
                                          float2 x1, float2 x2, float2 x3) {
  float2 acc = __fmul2_rn(w0, x0);
  acc = __ffma2_rn(w1, x1, acc);
  acc = __ffma2_rn(w2, x2, acc);
  acc = __ffma2_rn(w3, x3, acc);
  return acc;
}

// e^x with x clamped to [-87, 88], by Cody & Waite's reduction x = n ln2 + r
// (ln 2 split in a 16-bit high part, so n * high is exact, and a low part)
// and the degree-7 Taylor polynomial of e^r in Horner form, then scaling by
// 2^n. Every step is one correctly rounded IEEE operation, so any IEEE
// machine that follows the same steps gets the same bits: the post-conv
// activations, and hence their rounding to bf16, are reproducible. n is
// nearbyint(x * log2 e), obtained by adding and subtracting 1.5 * 2^23 (the
// add rounds to an integer); 2^n is built from the integer in t's low bits.
// Two values per call, with Blackwell's paired f32 instructions.
__device__ __forceinline__ float2 exp_cw2(float2 x) {
  constexpr float kMagic = 12582912.0f;                 // 1.5 * 2^23
  x.x = fminf(fmaxf(x.x, -87.0f), 88.0f);
  x.y = fminf(fmaxf(x.y, -87.0f), 88.0f);
  const float2 t = __fadd2_rn(__fmul2_rn(x, make_float2(1.44269504088896341f, 1.44269504088896341f)),
                              make_float2(kMagic, kMagic));
  const float2 n = __fadd2_rn(t, make_float2(-kMagic, -kMagic));
  const float2 mn = make_float2(-n.x, -n.y);
  float2 r = __ffma2_rn(mn, make_float2(0.693145751953125f, 0.693145751953125f), x);
  r = __ffma2_rn(mn, make_float2(1.42860682030941723212e-6f, 1.42860682030941723212e-6f), r);
  float2 p = make_float2(1.0f / 5040.0f, 1.0f / 5040.0f);
  p = __ffma2_rn(p, r, make_float2(1.0f / 720.0f, 1.0f / 720.0f));
  p = __ffma2_rn(p, r, make_float2(1.0f / 120.0f, 1.0f / 120.0f));
  p = __ffma2_rn(p, r, make_float2(1.0f / 24.0f, 1.0f / 24.0f));
  p = __ffma2_rn(p, r, make_float2(1.0f / 6.0f, 1.0f / 6.0f));
  p = __ffma2_rn(p, r, make_float2(0.5f, 0.5f));
  p = __ffma2_rn(p, r, make_float2(1.0f, 1.0f));
  p = __ffma2_rn(p, r, make_float2(1.0f, 1.0f));
  // 2^n: n sits in the low mantissa bits of t; (bits << 23) + bias is 2^n's pattern
  const float2 sc = make_float2(__int_as_float((__float_as_int(t.x) << 23) + 0x3f800000),
                                __int_as_float((__float_as_int(t.y) << 23) + 0x3f800000));
  return __fmul2_rn(p, sc);
}

// SiLU y / (1 + e^-y) with the exp above and an IEEE divide, two at a time.
__device__ __forceinline__ float2 silu2(float2 y) {
  const float2 d = __fadd2_rn(make_float2(1.0f, 1.0f), exp_cw2(make_float2(-y.x, -y.y)));
  return make_float2(__fdiv_rn(y.x, d.x), __fdiv_rn(y.y, d.y));
}

__device__ __forceinline__ float silu(float y) { return silu2(make_float2(y, 0.f)).x; }

// Sum of squares of a 128-channel head held as 8 contiguous channels by each
// of 16 consecutive lanes (lane & 15 = channel group). In-lane: strides 4, 2, 1;
// across lanes: xor 8, 4, 2, 1, which gives every lane the same bits because
// float addition is commutative. Must be called by all 32 lanes of the warp.
__device__ __forceinline__ float head_sum_sq16(const float v[8]) {
  const float2 e01 = __fmul2_rn(make_float2(v[0], v[1]), make_float2(v[0], v[1]));
  const float2 e23 = __fmul2_rn(make_float2(v[2], v[3]), make_float2(v[2], v[3]));
  const float2 e45 = __fmul2_rn(make_float2(v[4], v[5]), make_float2(v[4], v[5]));
  const float2 e67 = __fmul2_rn(make_float2(v[6], v[7]), make_float2(v[6], v[7]));
  const float2 p01 = __fadd2_rn(e01, e45);          // e0+e4, e1+e5
  const float2 p23 = __fadd2_rn(e23, e67);          // e2+e6, e3+e7
  const float2 q = __fadd2_rn(p01, p23);            // (p0+p2), (p1+p3)
  float g = __fadd_rn(q.x, q.y);
#pragma unroll
  for (int m = 8; m >= 1; m >>= 1) g = __fadd_rn(g, __shfl_xor_sync(FULL, g, m));
  return g;
}

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
