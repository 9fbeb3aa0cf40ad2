// Decode (the verify of T draft tokens with every token accepted, state and
// conv_state advanced in place) and the batched accepted-prefix commit across
// layers. The read-only verify is in verify.cu and follows the same order of
// arithmetic.
//
// Source: "Strata PR #3226" ("Summary": verify forward launched once per GDN
// layer; the 2-launch batched commit of conv_state and recurrent state across 36
// layers replacing 72 per-layer launches; committed states bitwise equal between
// the batched and per-layer routes) and the gated delta rule
// S_t = a_t S_{t-1}(I - b_t k_t k_t^T) + b_t v_t k_t^T, o_t = S_t q_t.
//
// Algorithm (derived from the rule; the pages give no formulas). Over the
// draft tokens t = 0..n-1 of one head, with r(t,s) = a_{s+1}...a_t (r(t,t) = 1)
// and g_t = a_0...a_t, the state after token t is
//     S_t = g_t S0 + sum_{s<=t} r(t,s) d_s k_s^T,
// where the deltas solve the unit lower-triangular system
//     d_t = b_t v_t - b_t g_t (S0 k_t) - sum_{s<t} b_t r(t,s) (k_t.k_s) d_s
// and the outputs are o_t = g_t (S0 q_t) + sum_{s<=t} r(t,s) (k_s.q_t) d_s.
// So S0 is read once and only 2T dot products per state row touch it (instead
// of 3T passes of the token-by-token form); the state write (commit) is one
// rank-n update. Value rows of S are independent, so each thread owns two rows
// x 32 columns of S0 in registers and the rows' deltas.
//
// One template body serves both modes, so the deltas and the committed state
// are computed by the same instructions in verify+commit and in decode: the
// bitwise agreement is by construction. No atomics, no inter-block waits.
//
// Global traffic goes out in the order the block waits on it: the gates and the
// conv's rows first, then the first v head's 64 KiB of state rows (issued before
// the small loads, the state read delayed them); the next head's state is asked
// into L2 early and its rows are loaded as soon as the current head's state is
// written, under the current head's epilogue.
//
// conv_state ownership: a block owns a whole q/k head group (the q and k heads
// and the Hv/Hk v heads that read them), so the block that reads a channel's
// conv_state rows is the only one that rewrites them, after a block barrier.
#include "common.cuh"
#include "launch.h"

namespace gdn {

enum StepMode { VERIFY_COMMIT_ALL = 1, COMMIT = 2, VERIFY_ONLY = 3 };

// Start bringing one head's 64 KiB state (contiguous in the pool) into L2: a
// hint, no completion to wait for.
__device__ __forceinline__ void prefetch_state_l2(const float* head_state) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(head_state), "r"(uint32_t(D * D * 4))
               : "memory");
}

constexpr int STEP_THREADS = 256;
constexpr int MAX_HEADS = 16;                    // v heads per block (Hv / Hk limit)


// Post-conv activation of 8 channels of draft token t: rows t..t+3 of
// (conv_state rows ++ draft rows), SiLU, then (q/k heads) the L2 norm, in f32:
// the recurrence takes them unrounded (they are never stored on this path).
// All 32 lanes of the warp must call it together.
template <int A>
__device__ __forceinline__ void draft_act8(const void* __restrict__ x_b, const void* __restrict__ cs,
                                           const void* __restrict__ conv_w, int C, int c, int t,
                                           bool live, bool is_qk, float eps, float v[8]) {
  float w[8][4];
  float rows[4][8];
  if (live) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float t8[8];
      load8<A>(conv_w, (int64_t)c * KW + 8 * q, t8);
#pragma unroll
      for (int j = 0; j < 8; ++j) w[2 * q + j / 4][j % 4] = t8[j];
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int idx = t + j;
      if (idx < KS) load8<A>(cs, (int64_t)idx * C + c, rows[j]);
      else load8<A>(x_b, (int64_t)(idx - KS) * C + c, rows[j]);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = silu(conv4(w[j], rows[0][j], rows[1][j], rows[2][j], rows[3][j]));
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = 0.f;
  }
  const float ss = head_sum_sq16(v);
  if (live && is_qk) {
    const float r = inv_norm(ss, eps);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __fmul_rn(v[j], r);
  }
}

// Warp dot product of two 128-vectors in shared memory; every lane gets the
// same bits (fixed in-lane order, then an xor butterfly).
__device__ __forceinline__ float warp_dot128(const float* a, const float* b) {
  const int lane = threadIdx.x & 31;
  const float4 x = reinterpret_cast<const float4*>(a)[lane];
  const float4 y = reinterpret_cast<const float4*>(b)[lane];
  float p = __fmul_rn(x.x, y.x);
  p = __fmaf_rn(x.y, y.y, p);
  p = __fmaf_rn(x.z, y.z, p);
  p = __fmaf_rn(x.w, y.w, p);
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) p = __fadd_rn(p, __shfl_xor_sync(FULL, p, m));
  return p;
}

// Dot products of the thread's two state rows (32 columns each, column
// 16m + 4cg + c) with a 128-vector in shared memory, completed over the 4 lanes
// that share the rows. All 4 lanes end with the same bits.
__device__ __forceinline__ void rows_dot(const float4 (&S)[2][8], const float* vec, int cg,
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

// One pass of the step over the draft tokens of sequence b = blockIdx.y of one
// layer, by MODE:
//   COMMIT             the first n_keep[b] tokens enter conv_state and state (no outputs)
//   VERIFY_COMMIT_ALL  outputs of the T tokens, conv_state and state advanced by all
//   VERIFY_ONLY        outputs of the T tokens, nothing written back
// The pass reads x, alpha, beta (T tokens per sequence) and the pools given, or
// with VIEWS those of layer blockIdx.z of the view table. Returns false when the
// sequence is skipped (padding, or a bad slot or n_keep, reported).
template <int A, int MODE, bool VIEWS>
__device__ __forceinline__ bool step_pass(const StepArgs& p, const void* x, const void* alpha,
                                          const void* beta, const int T, float* smem) {
  constexpr bool OUTPUTS = MODE != COMMIT;
  constexpr bool WRITES = MODE != VERIFY_ONLY;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.y;
  const int Hk = p.Hk, Hv = p.Hv, G = Hv / Hk;
  const int C = (2 * Hk + Hv) * D;

  const void* conv_w = p.conv_w;
  void* conv_state = p.conv_state;
  float* state = p.state;
  if constexpr (VIEWS) {                                  // the committing call walks the layers
    const gdn_layer_view lv = p.layers[blockIdx.z];
    x = lv.x; conv_w = lv.conv_w; conv_state = lv.conv_state; state = lv.state;
    alpha = lv.alpha; beta = lv.beta;
  }

  const int slot = p.slot_idx[b];
  if (slot < 0) return false;                             // padding entry
  if (slot >= p.n_slots) {
    if (tid == 0 && blockIdx.x == 0) report(p.dev_err, GDN_DEVERR_SLOT);
    return false;
  }
  int n = T;                                              // tokens that enter the state
  if constexpr (MODE == COMMIT) {
    n = p.n_keep[b];
    if (n < 0 || n > T) {
      if (tid == 0 && blockIdx.x == 0) report(p.dev_err, GDN_DEVERR_NKEEP);
      return false;
    }
    if (n == 0) return true;
  }

  // Heads of this block: a whole q/k head group.
  const int hq = blockIdx.x;                                       // q/k head
  const int h0 = blockIdx.x * G;                                   // first v head
  const int nh = G;                                                // v heads here

  // The first head's state rows (coalesced: 4 lanes cover 64 contiguous bytes of
  // a row; this thread owns rows 2rp, 2rp+1) go in flight after the small loads
  // the block waits on first: after the conv in decode and verify (7.53 -> 7.13 ms
  // per decode window), after the gates in the commit (0.914 -> 0.881 ms at
  // T = 8). Issued before them, the 64 KiB read delayed those loads.
  const int rp = tid >> 2, cg = tid & 3;
  const int row0 = 2 * rp;
  float4 S[2][8];
  auto load_first_state = [&]() {
    const float* Sg0 = state + (((int64_t)slot * Hv + h0) * D) * D;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
      for (int m = 0; m < 8; ++m)
        S[rr][m] = reinterpret_cast<const float4*>(Sg0 + (int64_t)(row0 + rr) * D)[4 * m + cg];
  };

  // shared memory: q[T][D], k[T][D], v[nh][T][D], o[T][D], small tables
  float* q_s = smem;
  float* k_s = q_s + MAXT * D;
  float* v_s = k_s + MAXT * D;
  float* o_s = v_s + (size_t)nh * MAXT * D;
  float* kk_s = o_s + MAXT * D;                  // [8][8] k_t . k_s
  float* qk_s = kk_s + MAXT * MAXT;              // [8][8] q_t . k_s
  float* A_s = qk_s + MAXT * MAXT;               // [8][8] b_t r(t,s) (k_t.k_s), s < t
  float* Oc_s = A_s + MAXT * MAXT;               // [8][8] r(t,s) (q_t.k_s), s <= t
  float* E_s = Oc_s + MAXT * MAXT;               // [8] r(n-1, s)
  float* g_s = E_s + MAXT;                       // [8] g_t
  float* bg_s = g_s + MAXT;                      // [8] b_t g_t
  float* b_s = bg_s + MAXT;                      // [8] b_t
  float* al_s = b_s + MAXT;                      // [nh][8] alpha of the block's heads
  float* be_s = al_s + MAXT * MAX_HEADS;         // [nh][8] beta

  const int64_t xb_off = (int64_t)b * T * C;
  const void* x_b = static_cast<const char*>(x) + xb_off * (A == BF16 ? 2 : 4);
  const int64_t cs_off = (int64_t)slot * KS * C;
  const void* cs = static_cast<const char*>(conv_state) + cs_off * (A == BF16 ? 2 : 4);

  // gates of the block's heads for the n tokens, staged once
  for (int e = tid; e < nh * n; e += STEP_THREADS) {
    const int g = e / n, t = e % n;
    const int64_t gi = ((int64_t)b * T + t) * Hv + h0 + g;
    const float ga = load_gate(alpha, gi, p.gate_bf16), gb = load_gate(beta, gi, p.gate_bf16);
    al_s[g * MAXT + t] = p.raw_gates ? gate_alpha(ga) : ga;      // raw projections: the gate step
    be_s[g * MAXT + t] = p.raw_gates ? gate_beta(gb) : gb;
  }

  if constexpr (MODE == COMMIT) load_first_state();

  // ---- phase 1: post-conv activations of the block's channels, tokens < n
  {
    const int groups_per_tok = (2 + nh) * 16;            // 8-channel groups per token
    const int items = n * groups_per_tok;
    const int iters = (items + STEP_THREADS - 1) / STEP_THREADS;
    for (int it = 0; it < iters; ++it) {
      const int item = it * STEP_THREADS + tid;
      const bool live = item < items;
      const int t = live ? item / groups_per_tok : 0;
      const int cgi = live ? item % groups_per_tok : 0;
      int c;                                             // global channel
      float* dst;
      bool is_qk;
      if (cgi < 16) { c = hq * D + cgi * 8; dst = q_s + t * D + cgi * 8; is_qk = true; }
      else if (cgi < 32) { c = (Hk + hq) * D + (cgi - 16) * 8; dst = k_s + t * D + (cgi - 16) * 8; is_qk = true; }
      else {
        const int g = (cgi - 32) >> 4, w8 = (cgi - 32) & 15;
        c = (2 * Hk + h0 + g) * D + w8 * 8;
        dst = v_s + ((size_t)g * MAXT + t) * D + w8 * 8;
        is_qk = false;
      }
      float v[8];
      draft_act8<A>(x_b, cs, conv_w, C, c, t, live, is_qk, p.eps, v);
      if (live) {
        reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
        if (OUTPUTS && p.postconv) store8<A>(p.postconv, xb_off + (int64_t)t * C + c, v);
      }
    }
  }
  __syncthreads();

  // ---- conv_state commit: last 3 rows of (old rows ++ draft rows 0..n-1)
  if constexpr (WRITES) {
    constexpr int MAXI = 4;                               // (2 + G) * 48 <= 4 * 256
    const int groups = (2 + nh) * 16;
    const int items = KS * groups;
    float keep[MAXI][8];
#pragma unroll
    for (int k = 0; k < MAXI; ++k) {
      const int item = k * STEP_THREADS + tid;
      if (item < items) {
        const int r = item / groups, cgi = item % groups;
        const int c = cgi < 32 ? (cgi < 16 ? hq * D + cgi * 8 : (Hk + hq) * D + (cgi - 16) * 8)
                               : (2 * Hk + h0 + ((cgi - 32) >> 4)) * D + ((cgi - 32) & 15) * 8;
        const int idx = n + r;
        if (idx < KS) load8<A>(cs, (int64_t)idx * C + c, keep[k]);
        else load8<A>(x_b, (int64_t)(idx - KS) * C + c, keep[k]);
      }
    }
    __syncthreads();                                      // every old row read first
#pragma unroll
    for (int k = 0; k < MAXI; ++k) {
      const int item = k * STEP_THREADS + tid;
      if (item < items) {
        const int r = item / groups, cgi = item % groups;
        const int c = cgi < 32 ? (cgi < 16 ? hq * D + cgi * 8 : (Hk + hq) * D + (cgi - 16) * 8)
                               : (2 * Hk + h0 + ((cgi - 32) >> 4)) * D + ((cgi - 32) & 15) * 8;
        store8<A>(conv_state, cs_off + (int64_t)r * C + c, keep[k]);
      }
    }
  }

  if constexpr (MODE != COMMIT) {
    load_first_state();
    // the second head's state into L2 while the first is computed (decode window
    // 7.15 -> 7.06 ms)
    if (tid == 0 && nh > 1) prefetch_state_l2(state + (((int64_t)slot * Hv + h0 + 1) * D) * D);
  }

  // ---- phase 2: key/key and query/key dot products (shared by the group); only
  // the pairs the tables use: k_t.k_s for s < t, q_t.k_s for s <= t
  for (int pr = warp; pr < 2 * MAXT * MAXT; pr += STEP_THREADS / 32) {
    const int which = pr / (MAXT * MAXT), t = (pr % (MAXT * MAXT)) / MAXT, s = pr % MAXT;
    if (t >= n || (which == 0 ? s >= t : s > t)) continue;   // warp-uniform
    if (which == 0) { const float d = warp_dot128(k_s + t * D, k_s + s * D); if (lane == 0) kk_s[t * MAXT + s] = d; }
    else if (OUTPUTS) { const float d = warp_dot128(q_s + t * D, k_s + s * D); if (lane == 0) qk_s[t * MAXT + s] = d; }
  }


  for (int g = 0; g < nh; ++g) {
    const int h = h0 + g;
    __syncthreads();                                      // kk/qk ready; tables free
    // gate tables for head h: one thread per (t, s), products in ascending
    // order (r(t,s) = a_{s+1} ... a_t, g_t = a_0 ... a_t)
    if (tid < MAXT * MAXT) {
      const int t = tid >> 3, sidx = tid & 7;
      if (t < n && sidx <= t) {
        const float* al = al_s + g * MAXT;
        float r = 1.f;
        for (int u = sidx + 1; u <= t; ++u) r = __fmul_rn(r, al[u]);
        const float bt = be_s[g * MAXT + t];
        if (sidx < t) A_s[t * MAXT + sidx] = __fmul_rn(__fmul_rn(bt, r), kk_s[t * MAXT + sidx]);
        if (OUTPUTS) Oc_s[t * MAXT + sidx] = __fmul_rn(r, qk_s[t * MAXT + sidx]);
        if (t == n - 1) E_s[sidx] = r;
        if (sidx == 0) {
          float gt = al[0];
          for (int u = 1; u <= t; ++u) gt = __fmul_rn(gt, al[u]);
          g_s[t] = gt;
          b_s[t] = bt;
          bg_s[t] = __fmul_rn(bt, gt);
        }
      }
    }
    // z of this head for the epilogue, in flight during the dot products
    Raw8<A> zraw;
    const int ep_t = tid >> 4, ep_l16 = tid & 15;
    const int64_t ep_zo = ((int64_t)b * T + ep_t) * Hv * D + (int64_t)h * D + ep_l16 * 8;
    if (OUTPUTS && tid < 128 && ep_t < n) raw_load<A>(p.z, ep_zo, zraw);
    // commit: the next head's state into L2 as each head starts (T = 8 commit
    // 0.883 -> 0.851 ms; earlier, with the first head's loads, was slower here)
    if constexpr (MODE == COMMIT) {
      if (tid == 0 && g + 1 < nh) prefetch_state_l2(state + (((int64_t)slot * Hv + h + 1) * D) * D);
    }
    // state rows of head h: in flight since load_first_state (head 0) or since the
    // previous head's state write (the others)
    float* Sg = state + (((int64_t)slot * Hv + h) * D) * D;
    __syncthreads();                                      // tables ready

    float d0[MAXT], d1[MAXT];
    const float* vh = v_s + (size_t)g * MAXT * D;
#pragma unroll
    for (int t = 0; t < MAXT; ++t) {
      if (t < n) {
        float sk0, sk1;
        rows_dot(S, k_s + t * D, cg, sk0, sk1);
        const float bt = b_s[t], bgt = bg_s[t];
        float r0 = __fmaf_rn(-bgt, sk0, __fmul_rn(bt, vh[t * D + row0]));
        float r1 = __fmaf_rn(-bgt, sk1, __fmul_rn(bt, vh[t * D + row0 + 1]));
#pragma unroll
        for (int s = 0; s < t; ++s) {
          const float a = A_s[t * MAXT + s];
          r0 = __fmaf_rn(-a, d0[s], r0);
          r1 = __fmaf_rn(-a, d1[s], r1);
        }
        d0[t] = r0;
        d1[t] = r1;
        if constexpr (OUTPUTS) {
          float sq0, sq1;
          rows_dot(S, q_s + t * D, cg, sq0, sq1);
          const float gt = g_s[t];
          float o0 = __fmul_rn(gt, sq0), o1 = __fmul_rn(gt, sq1);
#pragma unroll
          for (int s = 0; s <= t; ++s) {
            const float c = Oc_s[t * MAXT + s];
            o0 = __fmaf_rn(c, d0[s], o0);
            o1 = __fmaf_rn(c, d1[s], o1);
          }
          if (cg == 0) {
            o_s[t * D + row0] = __fmul_rn(o0, p.q_scale);
            o_s[t * D + row0 + 1] = __fmul_rn(o1, p.q_scale);
          }
        }
      }
    }

    // state commit: S_n = g_{n-1} S0 + sum_s r(n-1,s) d_s k_s^T, in place
    if constexpr (WRITES) {
      const float gl = g_s[n - 1];
      float e0[MAXT], e1[MAXT];
#pragma unroll
      for (int s = 0; s < MAXT; ++s) {
        if (s < n) { e0[s] = __fmul_rn(E_s[s], d0[s]); e1[s] = __fmul_rn(E_s[s], d1[s]); }
      }
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        float4 a = S[0][m], c = S[1][m];
        a.x = __fmul_rn(gl, a.x); a.y = __fmul_rn(gl, a.y); a.z = __fmul_rn(gl, a.z); a.w = __fmul_rn(gl, a.w);
        c.x = __fmul_rn(gl, c.x); c.y = __fmul_rn(gl, c.y); c.z = __fmul_rn(gl, c.z); c.w = __fmul_rn(gl, c.w);
#pragma unroll
        for (int s = 0; s < MAXT; ++s) {
          if (s < n) {
            const float4 k = reinterpret_cast<const float4*>(k_s + s * D)[4 * m + cg];
            a.x = __fmaf_rn(e0[s], k.x, a.x); a.y = __fmaf_rn(e0[s], k.y, a.y);
            a.z = __fmaf_rn(e0[s], k.z, a.z); a.w = __fmaf_rn(e0[s], k.w, a.w);
            c.x = __fmaf_rn(e1[s], k.x, c.x); c.y = __fmaf_rn(e1[s], k.y, c.y);
            c.z = __fmaf_rn(e1[s], k.z, c.z); c.w = __fmaf_rn(e1[s], k.w, c.w);
          }
        }
        reinterpret_cast<float4*>(Sg + (int64_t)row0 * D)[4 * m + cg] = a;
        reinterpret_cast<float4*>(Sg + (int64_t)(row0 + 1) * D)[4 * m + cg] = c;
      }
    }
    if (g + 1 < nh) {                                     // the next head's rows go in flight now,
      const float* Sn = Sg + (int64_t)D * D;              // under this head's epilogue
#pragma unroll
      for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int m = 0; m < 8; ++m)
          S[rr][m] = reinterpret_cast<const float4*>(Sn + (int64_t)(row0 + rr) * D)[4 * m + cg];
    }

    // z-gated RMSNorm of the outputs: one 16-lane group per token
    if constexpr (OUTPUTS) {
      __syncthreads();                                    // o_s complete
      if (tid < 128) {                                    // warps 0..3 take part fully
        const int t = tid >> 4, l16 = tid & 15;
        const bool live = t < n;
        float o[8];
        if (live) {
          const float4 u0 = reinterpret_cast<const float4*>(o_s + t * D)[2 * l16];
          const float4 u1 = reinterpret_cast<const float4*>(o_s + t * D)[2 * l16 + 1];
          o[0] = u0.x; o[1] = u0.y; o[2] = u0.z; o[3] = u0.w;
          o[4] = u1.x; o[5] = u1.y; o[6] = u1.z; o[7] = u1.w;
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) o[j] = 0.f;
        }
        const float ss = head_sum_sq16(o);
        if (live) {
          const float r = inv_norm(__fmul_rn(ss, 1.0f / D), p.eps);
          const int64_t zo = ep_zo;
          float zv[8], res[8];
          raw_unpack<A>(zraw, zv);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            res[j] = __fmul_rn(__fmul_rn(__fmul_rn(o[j], r), p.norm_w[l16 * 8 + j]), silu_gate(zv[j]));
          store_out8<A>(p.out, zo, res, p.out_f32);
        }
      }
    }
  }
  return true;
}

template <int A, int MODE>
__global__ void __launch_bounds__(STEP_THREADS, 2) step_kernel(StepArgs p) {
  extern __shared__ __align__(16) float smem[];
  step_pass<A, MODE, MODE == COMMIT>(p, p.x, p.alpha, p.beta, p.T, smem);
}

// Verify with the previous window's commit folded in: first the accepted
// prefix (n_keep[b] of its prev_T tokens) of the previous window enters
// conv_state and state, by the same instructions as the batched commit, then
// the T new draft tokens are verified from the committed state, which this
// block has just written (its state rows come back from L2; each thread reads
// the rows it wrote). Nothing of the new drafts is written back.
template <int A>
__global__ void __launch_bounds__(STEP_THREADS, 2) lazy_kernel(StepArgs p) {
  extern __shared__ __align__(16) float smem[];
  if (!step_pass<A, COMMIT, false>(p, p.prev_x, p.prev_alpha, p.prev_beta, p.prev_T, smem)) return;
  __syncthreads();                                        // conv_state rows and tables settled
  step_pass<A, VERIFY_ONLY, false>(p, p.x, p.alpha, p.beta, p.T, smem);
}

size_t step_smem_bytes(int nh) {
  return sizeof(float) * ((size_t)(3 + nh) * MAXT * D + 4 * MAXT * MAXT + 4 * MAXT +
                          2 * MAXT * MAX_HEADS);
}

// Decode and the batched commit run the same body on the CUDA cores (n accepted
// key dots per state row, no query dots for the commit), so decode and
// verify + commit leave bitwise equal states.
template <int A, int MODE>
static cudaError_t launch_mode(const StepArgs& a, dim3 grid, int nh, cudaStream_t stream) {
  const size_t smem = step_smem_bytes(nh);
  if (smem > 48 * 1024) {
    cudaError_t e = set_smem_once<step_kernel<A, MODE>>((int)smem);
    if (e != cudaSuccess) return e;
  }
  step_kernel<A, MODE><<<grid, STEP_THREADS, smem, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_verify(const StepArgs& a, bool commit_all, int act, cudaStream_t stream) {
  if (!commit_all) return launch_verify_readonly(a, act, stream);
  dim3 grid(a.Hk, a.B, 1);
  const int nh = a.Hv / a.Hk;
  return act == GDN_BF16 ? launch_mode<BF16, VERIFY_COMMIT_ALL>(a, grid, nh, stream)
                         : launch_mode<F32, VERIFY_COMMIT_ALL>(a, grid, nh, stream);
}

template <int A>
static cudaError_t launch_lazy_t(const StepArgs& a, cudaStream_t stream) {
  const int nh = a.Hv / a.Hk;
  const size_t smem = step_smem_bytes(nh);
  if (smem > 48 * 1024) {
    cudaError_t e = set_smem_once<lazy_kernel<A>>((int)smem);
    if (e != cudaSuccess) return e;
  }
  lazy_kernel<A><<<dim3(a.Hk, a.B, 1), STEP_THREADS, smem, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_verify_lazy(const StepArgs& a, int act, cudaStream_t stream) {
  return act == GDN_BF16 ? launch_lazy_t<BF16>(a, stream) : launch_lazy_t<F32>(a, stream);
}

cudaError_t launch_commit(const StepArgs& a, int L, int act, cudaStream_t stream) {
  dim3 grid(a.Hk, a.B, L);
  const int nh = a.Hv / a.Hk;
  return act == GDN_BF16 ? launch_mode<BF16, COMMIT>(a, grid, nh, stream)
                         : launch_mode<F32, COMMIT>(a, grid, nh, stream);
}

}  // namespace gdn
