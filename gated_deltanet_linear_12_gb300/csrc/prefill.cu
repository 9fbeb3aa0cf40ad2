// Chunked (WY-form) gated delta rule over varlen sequences, 64-token chunks,
// with the z-gated RMSNorm fused into the output. CUDA-core (FFMA) version:
// every product is an f32 FMA; this is the f32-activation path and the
// reference route for the tensor-core path.
//
// Source: the rule S_t = a_t S_{t-1}(I - b_t k_t k_t^T) + b_t v_t k_t^T,
// o_t = S_t q_t, and the output norm after the recurrence ("Strata PR #3226").
// Within a chunk (chunk-local g_t = sum_{u<=t} log a_u, G_t = exp(g_t)):
//   A_ts = b_t exp(g_t - g_s) (k_t . k_s)  (s < t),   Tinv = (I + A)^-1
//   R_t  = b_t v_t - b_t G_t (S0 k_t)                  D = Tinv R   (the deltas)
//   O_t  = G_t (S0 q_t) + sum_{s<=t} exp(g_t - g_s) (q_t . k_s) D_s
//   S    = G_last S0 + sum_s exp(g_last - g_s) D_s k_s^T
// A partial last chunk is padded with k = q = v = 0, b = 0, a = 1, which is an
// exact identity step. One block per (sequence, v head) walks the sequence's
// chunks with S0 resident in registers (two value rows x 32 key columns per
// thread), so the state never leaves the SM between chunks.
#include "common.cuh"
#include "launch.h"

namespace gdn {

constexpr int PF_THREADS = 256;
constexpr int DP = D + 4;          // padded row stride of [64][128] tiles (conflict-free LDS.128)
constexpr int XP = CHUNK + 1;      // padded row stride of [64][64] tiles


size_t prefill_smem_bytes() {
  return sizeof(float) * ((size_t)5 * CHUNK * DP + 2 * CHUNK * XP + 4 * CHUNK);
}

// acc[i][c] (+)= sum_s L[row_i][s] * M[s][col_c] over s < 64, for rows
// ty + 16 i (i < 4) and columns 4 tx + {0..3} + 64 {0,1}; L has stride XP and
// M stride DP.
__device__ __forceinline__ void tile_lm(const float* L, const float* M, int ty, int tx,
                                        float acc[4][8]) {
#pragma unroll 4
  for (int s = 0; s < CHUNK; ++s) {
    const float4 m0 = reinterpret_cast<const float4*>(M + s * DP)[tx];
    const float4 m1 = reinterpret_cast<const float4*>(M + s * DP + 64)[tx];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float l = L[(ty + 16 * i) * XP + s];
      acc[i][0] = __fmaf_rn(l, m0.x, acc[i][0]); acc[i][1] = __fmaf_rn(l, m0.y, acc[i][1]);
      acc[i][2] = __fmaf_rn(l, m0.z, acc[i][2]); acc[i][3] = __fmaf_rn(l, m0.w, acc[i][3]);
      acc[i][4] = __fmaf_rn(l, m1.x, acc[i][4]); acc[i][5] = __fmaf_rn(l, m1.y, acc[i][5]);
      acc[i][6] = __fmaf_rn(l, m1.z, acc[i][6]); acc[i][7] = __fmaf_rn(l, m1.w, acc[i][7]);
    }
  }
}

// X[t][s] = P[t] . Q[s] for t = ty + 16 i, s = tx + 16 c (P, Q stride DP).
__device__ __forceinline__ void gram(const float* P, const float* Q, float* X, int ty, int tx) {
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[i][c] = 0.f;
#pragma unroll 4
  for (int j = 0; j < D; j += 4) {
    float4 pv[4], qv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) pv[i] = *reinterpret_cast<const float4*>(P + (ty + 16 * i) * DP + j);
#pragma unroll
    for (int c = 0; c < 4; ++c) qv[c] = *reinterpret_cast<const float4*>(Q + (tx + 16 * c) * DP + j);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        acc[i][c] = __fmaf_rn(pv[i].x, qv[c].x, acc[i][c]);
        acc[i][c] = __fmaf_rn(pv[i].y, qv[c].y, acc[i][c]);
        acc[i][c] = __fmaf_rn(pv[i].z, qv[c].z, acc[i][c]);
        acc[i][c] = __fmaf_rn(pv[i].w, qv[c].w, acc[i][c]);
      }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int c = 0; c < 4; ++c) X[(ty + 16 * i) * XP + tx + 16 * c] = acc[i][c];
}

// Dot products of the thread's two state rows with a 128-vector (row of a DP
// tile), completed over the 4 lanes that share the rows.
__device__ __forceinline__ void rows_dot_pf(const float4 (&S)[2][8], const float* vec, int cg,
                                            float& r0, float& r1) {
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const float4 k = reinterpret_cast<const float4*>(vec)[4 * m + cg];
    a0 = __fmaf_rn(S[0][m].x, k.x, a0); a0 = __fmaf_rn(S[0][m].y, k.y, a0);
    a0 = __fmaf_rn(S[0][m].z, k.z, a0); a0 = __fmaf_rn(S[0][m].w, k.w, a0);
    a1 = __fmaf_rn(S[1][m].x, k.x, a1); a1 = __fmaf_rn(S[1][m].y, k.y, a1);
    a1 = __fmaf_rn(S[1][m].z, k.z, a1); a1 = __fmaf_rn(S[1][m].w, k.w, a1);
  }
  a0 = __fadd_rn(a0, __shfl_xor_sync(FULL, a0, 1));
  a1 = __fadd_rn(a1, __shfl_xor_sync(FULL, a1, 1));
  a0 = __fadd_rn(a0, __shfl_xor_sync(FULL, a0, 2));
  a1 = __fadd_rn(a1, __shfl_xor_sync(FULL, a1, 2));
  r0 = a0;
  r1 = a1;
}

template <int A>
__global__ void __launch_bounds__(PF_THREADS, 1) prefill_ffma_kernel(PrefillArgs p) {
  extern __shared__ __align__(16) float smem[];
  float* Ks = smem;                       // [64][DP] keys
  float* Qs = Ks + CHUNK * DP;            // [64][DP] queries
  float* Vs = Qs + CHUNK * DP;            // [64][DP] values
  float* Rs = Vs + CHUNK * DP;            // [64][DP] rhs -> S0 q -> outputs
  float* Ds = Rs + CHUNK * DP;            // [64][DP] deltas (first: inverse scratch)
  float* Xs = Ds + CHUNK * DP;            // [64][XP] k.k -> A -> scaled q.k
  float* Ys = Xs + CHUNK * XP;            // [64][XP] (I + A)^-1
  float* gl_s = Ys + CHUNK * XP;          // [64] g_t (chunk-local log decay)
  float* G_s = gl_s + CHUNK;              // [64] exp(g_t)
  float* b_s = G_s + CHUNK;               // [64] beta
  float* c_s = b_s + CHUNK;               // [64] exp(g_last - g_t)

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x, s = blockIdx.y;
  const int Hk = p.Hk, Hv = p.Hv, hq = h / (Hv / Hk);
  const int C = (2 * Hk + Hv) * D;
  const int slot = p.slot_idx[s];
  if (slot < 0) return;
  if (slot >= p.n_slots) {
    if (tid == 0 && h == 0) report(p.dev_err, GDN_DEVERR_SLOT);
    return;
  }
  const int64_t seq0 = p.cu[s], seq1 = p.cu[s + 1];
  if (seq1 < seq0 || seq0 < 0 || seq1 > p.n_tok) {
    if (tid == 0 && h == 0) report(p.dev_err, GDN_DEVERR_SEQLENS);
    return;
  }
  const int rp = tid >> 2, cg = tid & 3, row0 = 2 * rp;   // state rows of this thread
  const int ty = tid >> 4, tx = tid & 15;                 // tile coordinates

  float* Sg = p.state + (((int64_t)slot * Hv + h) * D) * D;
  float4 S[2][8];
  if (p.has_init[s]) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
      for (int m = 0; m < 8; ++m)
        S[rr][m] = reinterpret_cast<const float4*>(Sg + (int64_t)(row0 + rr) * D)[4 * m + cg];
  } else {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
      for (int m = 0; m < 8; ++m) S[rr][m] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  for (int64_t c0 = seq0; c0 < seq1; c0 += CHUNK) {
    const int m = (int)(seq1 - c0 < CHUNK ? seq1 - c0 : CHUNK);
    // ---- load the chunk (zero / identity padding past m)
    for (int it = tid; it < CHUNK * 48; it += PF_THREADS) {
      const int t = it / 48, part = it % 48, which = part / 16, w8 = part % 16;
      float v[8];
      if (t < m) {
        const int ch = which == 0 ? hq * D : (which == 1 ? (Hk + hq) * D : (2 * Hk + h) * D);
        load8<A>(p.qkv, (c0 + t) * C + ch + w8 * 8, v);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = 0.f;
      }
      float* dst = (which == 0 ? Qs : (which == 1 ? Ks : Vs)) + t * DP + w8 * 8;
      reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
      reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
    if (warp == 0) {                       // chunk-local log-decay scan (2 tokens per lane)
      const int t0 = 2 * lane;
      // raw projections: the gate step on the values read
      auto alpha_of = [&](int64_t gi) { const float v = load_gate(p.alpha, gi, p.gate_bf16); return p.raw_gates ? gate_alpha(v) : v; };
      auto beta_of = [&](int64_t gi) { const float v = load_gate(p.beta, gi, p.gate_bf16); return p.raw_gates ? gate_beta(v) : v; };
      const float la0 = t0 < m ? logf(alpha_of((c0 + t0) * Hv + h)) : 0.f;
      const float la1 = t0 + 1 < m ? logf(alpha_of((c0 + t0 + 1) * Hv + h)) : 0.f;
      const float pair = la0 + la1;
      float inc = pair;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float v = __shfl_up_sync(FULL, inc, o);
        if (lane >= o) inc += v;
      }
      const float g0 = inc - pair + la0, g1 = inc;
      gl_s[t0] = g0;
      gl_s[t0 + 1] = g1;
      b_s[t0] = t0 < m ? beta_of((c0 + t0) * Hv + h) : 0.f;
      b_s[t0 + 1] = t0 + 1 < m ? beta_of((c0 + t0 + 1) * Hv + h) : 0.f;
      const float glast = __shfl_sync(FULL, g1, 31);
      G_s[t0] = expf(g0);
      G_s[t0 + 1] = expf(g1);
      c_s[t0] = expf(glast - g0);
      c_s[t0 + 1] = expf(glast - g1);
    }
    __syncthreads();

    // ---- A = strictly lower (b_t exp(g_t - g_s) k_t.k_s)
    gram(Ks, Ks, Xs, ty, tx);
    __syncthreads();
    for (int e = tid; e < CHUNK * CHUNK; e += PF_THREADS) {
      const int t = e / CHUNK, u = e % CHUNK;
      float a = 0.f;
      if (u < t) a = b_s[t] * expf(gl_s[t] - gl_s[u]) * Xs[t * XP + u];
      Xs[t * XP + u] = a;
      Ys[t * XP + u] = 0.f;
    }
    __syncthreads();
    // ---- Tinv = (I + A)^-1 by recursive doubling over 16/32/64 blocks
    if (tid < CHUNK) {                     // 16x16 diagonal blocks, one column per thread
      const int j = tid, blk = j & ~15;
      Ys[j * XP + j] = 1.f;
      for (int t = j + 1; t < blk + 16; ++t) {
        float acc = 0.f;
        for (int u = j; u < t; ++u) acc = __fmaf_rn(Xs[t * XP + u], Ys[u * XP + j], acc);
        Ys[t * XP + j] = -acc;
      }
    }
    __syncthreads();
    float* tmp = Ds;                       // scratch [32][32] (stride 32)
    // level 2: for each 32-block P, Y[16+i][j] = -Y22 (A21 Y11), i,j < 16
    {
      const int P = tid >> 7, e = tid & 127;          // 2 blocks x 256 entries, 2 per thread
      for (int k = 0; k < 2; ++k) {
        const int ent = e * 2 + k, i = ent >> 4, j = ent & 15, base = 32 * P;
        float acc = 0.f;
        for (int u = 0; u < 16; ++u)
          acc = __fmaf_rn(Xs[(base + 16 + i) * XP + base + u], Ys[(base + u) * XP + base + j], acc);
        tmp[P * 256 + ent] = acc;
      }
    }
    __syncthreads();
    {
      const int P = tid >> 7, e = tid & 127;
      for (int k = 0; k < 2; ++k) {
        const int ent = e * 2 + k, i = ent >> 4, j = ent & 15, base = 32 * P;
        float acc = 0.f;
        for (int u = 0; u < 16; ++u)
          acc = __fmaf_rn(Ys[(base + 16 + i) * XP + base + 16 + u], tmp[P * 256 + u * 16 + j], acc);
        Ys[(base + 16 + i) * XP + base + j] = -acc;
      }
    }
    __syncthreads();
    // level 3: Y[32+i][j] = -Y[32:,32:] (A[32:,:32] Y[:32,:32]), i,j < 32
    for (int k = 0; k < 4; ++k) {
      const int ent = tid * 4 + k, i = ent >> 5, j = ent & 31;
      float acc = 0.f;
      for (int u = j & ~15; u < 32; ++u)                       // Y[u][j] = 0 for u < j's block
        acc = __fmaf_rn(Xs[(32 + i) * XP + u], Ys[u * XP + j], acc);
      tmp[ent] = acc;
    }
    __syncthreads();
    for (int k = 0; k < 4; ++k) {
      const int ent = tid * 4 + k, i = ent >> 5, j = ent & 31;
      float acc = 0.f;
      for (int u = 0; u <= i; ++u)
        acc = __fmaf_rn(Ys[(32 + i) * XP + 32 + u], tmp[u * 32 + j], acc);
      Ys[(32 + i) * XP + j] = -acc;
    }
    __syncthreads();

    // ---- R = b v - b G (S0 k)
    for (int t = 0; t < CHUNK; ++t) {
      float sk0, sk1;
      rows_dot_pf(S, Ks + t * DP, cg, sk0, sk1);
      if (cg == 0) {
        const float bt = b_s[t], bg = __fmul_rn(bt, G_s[t]);
        Rs[t * DP + row0] = __fmaf_rn(-bg, sk0, __fmul_rn(bt, Vs[t * DP + row0]));
        Rs[t * DP + row0 + 1] = __fmaf_rn(-bg, sk1, __fmul_rn(bt, Vs[t * DP + row0 + 1]));
      }
    }
    __syncthreads();
    // ---- D = Tinv R
    {
      float acc[4][8];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[i][c] = 0.f;
      tile_lm(Ys, Rs, ty, tx, acc);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float* d = Ds + (ty + 16 * i) * DP;
        reinterpret_cast<float4*>(d)[tx] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        reinterpret_cast<float4*>(d + 64)[tx] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
      }
    }
    __syncthreads();
    // ---- S0 q into R, q.k into X (scaled, causal)
    for (int t = 0; t < CHUNK; ++t) {
      float sq0, sq1;
      rows_dot_pf(S, Qs + t * DP, cg, sq0, sq1);
      if (cg == 0) {
        Rs[t * DP + row0] = __fmul_rn(G_s[t], sq0);
        Rs[t * DP + row0 + 1] = __fmul_rn(G_s[t], sq1);
      }
    }
    gram(Qs, Ks, Xs, ty, tx);
    __syncthreads();
    for (int e = tid; e < CHUNK * CHUNK; e += PF_THREADS) {
      const int t = e / CHUNK, u = e % CHUNK;
      Xs[t * XP + u] = u <= t ? expf(gl_s[t] - gl_s[u]) * Xs[t * XP + u] : 0.f;
    }
    __syncthreads();
    // ---- O = G (S0 q) + X D  (in place in R)
    {
      float acc[4][8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 r0 = reinterpret_cast<const float4*>(Rs + (ty + 16 * i) * DP)[tx];
        const float4 r1 = reinterpret_cast<const float4*>(Rs + (ty + 16 * i) * DP + 64)[tx];
        acc[i][0] = r0.x; acc[i][1] = r0.y; acc[i][2] = r0.z; acc[i][3] = r0.w;
        acc[i][4] = r1.x; acc[i][5] = r1.y; acc[i][6] = r1.z; acc[i][7] = r1.w;
      }
      tile_lm(Xs, Ds, ty, tx, acc);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float* d = Rs + (ty + 16 * i) * DP;
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[i][c] = __fmul_rn(acc[i][c], p.q_scale);
        reinterpret_cast<float4*>(d)[tx] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        reinterpret_cast<float4*>(d + 64)[tx] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
      }
    }
    // ---- S = G_last S0 + sum_s c_s D_s k_s^T   (registers; reads D, K only)
    {
      const float gl = G_s[CHUNK - 1];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int mm = 0; mm < 8; ++mm) {
          S[rr][mm].x = __fmul_rn(gl, S[rr][mm].x); S[rr][mm].y = __fmul_rn(gl, S[rr][mm].y);
          S[rr][mm].z = __fmul_rn(gl, S[rr][mm].z); S[rr][mm].w = __fmul_rn(gl, S[rr][mm].w);
        }
      for (int u = 0; u < CHUNK; ++u) {
        const float cu = c_s[u];
        const float e0 = __fmul_rn(cu, Ds[u * DP + row0]);
        const float e1 = __fmul_rn(cu, Ds[u * DP + row0 + 1]);
#pragma unroll
        for (int mm = 0; mm < 8; ++mm) {
          const float4 k = reinterpret_cast<const float4*>(Ks + u * DP)[4 * mm + cg];
          S[0][mm].x = __fmaf_rn(e0, k.x, S[0][mm].x); S[0][mm].y = __fmaf_rn(e0, k.y, S[0][mm].y);
          S[0][mm].z = __fmaf_rn(e0, k.z, S[0][mm].z); S[0][mm].w = __fmaf_rn(e0, k.w, S[0][mm].w);
          S[1][mm].x = __fmaf_rn(e1, k.x, S[1][mm].x); S[1][mm].y = __fmaf_rn(e1, k.y, S[1][mm].y);
          S[1][mm].z = __fmaf_rn(e1, k.z, S[1][mm].z); S[1][mm].w = __fmaf_rn(e1, k.w, S[1][mm].w);
        }
      }
    }
    __syncthreads();
    // ---- z-gated RMSNorm of the outputs, one 16-lane group per token
    for (int it = 0; it < CHUNK / (PF_THREADS / 16); ++it) {
      const int t = it * (PF_THREADS / 16) + (tid >> 4), l16 = tid & 15;
      const bool live = t < m;
      float o[8];
      const float4 u0 = reinterpret_cast<const float4*>(Rs + t * DP)[2 * l16];
      const float4 u1 = reinterpret_cast<const float4*>(Rs + t * DP)[2 * l16 + 1];
      o[0] = u0.x; o[1] = u0.y; o[2] = u0.z; o[3] = u0.w;
      o[4] = u1.x; o[5] = u1.y; o[6] = u1.z; o[7] = u1.w;
      const float ss = head_sum_sq16(o);
      if (live) {
        const float r = inv_norm(__fmul_rn(ss, 1.0f / D), p.eps);
        const int64_t zo = (c0 + t) * Hv * D + (int64_t)h * D + l16 * 8;
        float zv[8], res[8];
        load8<A>(p.z, zo, zv);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          res[j] = __fmul_rn(__fmul_rn(__fmul_rn(o[j], r), p.norm_w[l16 * 8 + j]), silu_gate(zv[j]));
        store_out8<A>(p.out, zo, res, p.out_f32);
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int rr = 0; rr < 2; ++rr)
#pragma unroll
    for (int mm = 0; mm < 8; ++mm)
      reinterpret_cast<float4*>(Sg + (int64_t)(row0 + rr) * D)[4 * mm + cg] = S[rr][mm];
}

cudaError_t launch_prefill(const PrefillArgs& a, int act, cudaStream_t stream) {
  if (act == GDN_BF16) return launch_prefill_tc(a, stream);   // tensor-core path
  const size_t smem = prefill_smem_bytes();
  dim3 grid(a.Hv, a.n_seq);
  cudaError_t e;
  if (act == GDN_BF16) {
    e = cudaFuncSetAttribute(prefill_ffma_kernel<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prefill_ffma_kernel<BF16><<<grid, PF_THREADS, smem, stream>>>(a);
  } else {
    e = cudaFuncSetAttribute(prefill_ffma_kernel<F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prefill_ffma_kernel<F32><<<grid, PF_THREADS, smem, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace gdn
