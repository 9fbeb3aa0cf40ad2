// Chunked (WY-form) gated delta rule over varlen sequences on the 5th-gen
// tensor cores (bf16 activations), 64-token chunks, z-gated RMSNorm fused.
//
// Source: the rule S_t = a_t S_{t-1}(I - b_t k_t k_t^T) + b_t v_t k_t^T,
// o_t = S_t q_t, and the output norm after the recurrence ("Strata PR #3226").
// Per chunk (chunk-local g_t = sum_{u<=t} log a_u, G_t = e^{g_t},
// c_t = e^{g_last - g_t}):
//   A_ts = b_t e^{g_t - g_s} k_t.k_s (s < t),     (I + A) d = R
//   R_t  = b_t v_t - b_t G_t S0 k_t
//   o_t  = G_t S0 q_t + sum_{s<=t} e^{g_t - g_s} (q_t.k_s) d_s
//   S    = G_last S0 + sum_s c_s d_s k_s^T
// Written transposed, value row i of S is TMEM lane i and the products are
//   MMA1  P^T  = S0 [K;Q]^T     M=128 N=128 K=128   S0 as bf16 hi + lo (2 passes)
//   MMA2  G    = [K;Q] K^T      M=128 N=64  K=128   exact bf16 products
//   MMA5  O^T  = D^T X^T        M=128 N=64  K=64    3 passes (hi hi, lo hi, hi lo)
//   MMA3  dS   = (c D)^T K      M=128 N=128 K=64    (c D) as hi + lo (2 passes)
// where X_ts = e^{g_t - g_s} q_t.k_s (s <= t). An f32 operand x enters as
// hi = bf16(x), lo = bf16(x - hi): the dropped lo*lo term and the rounding of
// lo leave a relative error near 2^-16 per product, far below the 1e-4 bound
// on states. S stays in f32 in TMEM for the whole sequence; only its bf16
// hi/lo copies (MMA operands) are rewritten per chunk. CUDA cores build the
// decay tables and solve (I + A) d = R for each value row by forward
// substitution in f32 (the row's R and d stay in one thread's registers),
// while the other half of the block runs the previous chunk's RMSNorm.
// One block of 256 threads per (sequence, v head); warps w and w + 4 share
// TMEM lane quarter w % 4 (rows i = 32 (w % 4) + lane). Every wait is bounded.
#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace gdn {

namespace {

constexpr int PT = 256;
constexpr int C64 = CHUNK;           // 64
constexpr int AP = C64 + 4;          // row stride of the f32 64x64 tables (16-byte rows)

// shared memory map (bytes); K-major tiles use tc::kmajor_offset
constexpr int SM_SHI = 0;                          // S hi   128x128 bf16 (MMA1 A)
constexpr int SM_SLO = SM_SHI + 32768;             // S lo
constexpr int SM_KQ = SM_SLO + 32768;              // [K;Q]  128x128 bf16 (MMA1 B, MMA2 A and B);
                                                   // then (cD)^T hi | lo, 128x64 each (MMA3 A)
constexpr int SM_KT = SM_KQ + 32768;               // K^T    128x64 bf16 (MMA3 B)
constexpr int SM_RD = SM_KT + 16384;               // D^T hi | lo, 128x64 each (MMA5 A);
                                                   // then outputs [64][128] f32
constexpr int SM_TI = SM_RD + 32768;               // the chunk's values [64][128] bf16
constexpr int SM_XB = SM_TI + 16384;               // X hi | lo, 64x64 each (MMA5 B)
constexpr int SM_AB = SM_XB + 16384;               // A^T f32 [64][AP]: column u of A is row u
constexpr int SM_ZB = SM_AB + 64 * AP * 4;         // the previous chunk's z rows [64][128] bf16
constexpr int SM_VEC = SM_ZB + 16384;              // g2, G, b, c, la [64] f32
constexpr int SM_BAR = SM_VEC + 5 * 64 * 4;        // MMA mbarrier (8 B), TMEM slot, rank pick,
constexpr int SM_TOTAL = SM_BAR + 24;              // row-tile mbarrier (8 B at +16)

constexpr uint32_t TM_COLS = 512;
constexpr uint32_t TM_S = 0;         // S f32                    cols   0..127
constexpr uint32_t TM_P = 128;       // P^T = [S0 k | S0 q]      cols 128..255
constexpr uint32_t TM_G = 256;       // G = [K;Q] K^T            cols 256..319
constexpr uint32_t TM_DS = 256;      // dS (after G is read)     cols 256..383
constexpr uint32_t TM_O = 384;       // O^T                      cols 384..447
constexpr uint32_t WAIT_POLLS = 1u << 24;

__device__ __forceinline__ void st16(uint8_t* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// 2^x by the hardware approximation (relative error about 2^-22).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

using tc::cp_async16;
using tc::cp_async4;
using tc::cp_async_commit;
using tc::cp_async_wait_all;

// One row (K = 64 values) of a K-major tile with `rows` rows, as bf16 hi | lo.
__device__ __forceinline__ void put_row64(uint8_t* hi_tile, uint8_t* lo_tile, int row, int rows,
                                          const float* x) {
#pragma unroll
  for (int q8 = 0; q8 < 8; ++q8) {
    uint4 hi, lo;
    tc::split8(x + 8 * q8, hi, lo);
    st16(hi_tile + tc::kmajor_offset(row, 8 * q8, rows), hi);
    st16(lo_tile + tc::kmajor_offset(row, 8 * q8, rows), lo);
  }
}

// n_slices K=16 slices of one MMA pass over K-major tiles of a_rows / b_rows
// rows (the K-slice stride is two core-matrix columns: 2 * rows/8 * 128 bytes).
__device__ __forceinline__ void mma_pass(uint32_t d_tmem, uint32_t a, int a_rows, uint32_t b,
                                         int b_rows, int n_slices, uint32_t idesc, bool acc_first) {
  const uint32_t a_lbo = (uint32_t)(a_rows / 8) * 128, b_lbo = (uint32_t)(b_rows / 8) * 128;
#pragma unroll 1
  for (int ks = 0; ks < n_slices; ++ks)
    tc::mma_bf16(d_tmem, tc::smem_desc(a + ks * 2 * a_lbo, a_lbo, 128),
                 tc::smem_desc(b + ks * 2 * b_lbo, b_lbo, 128), idesc,
                 (acc_first || ks > 0) ? 1u : 0u);
}

}  // namespace

// 2-D TMA copy of a box of a row-major bf16 tensor (x = column, y = row).
__device__ __forceinline__ void tma_rows(uint8_t* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          tc::smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(tc::smem_u32(bar))
      : "memory");
}

// vmap: the qkv rows [n_tok][C], zmap: the z rows [n_tok][Hv * 128], both in
// boxes of 128 columns x 64 rows (one head of one chunk).
__global__ void __launch_bounds__(PT, 1)
prefill_tc_kernel(PrefillArgs p, const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap zmap) {
  extern __shared__ __align__(1024) uint8_t sm[];
  uint8_t* SHI = sm + SM_SHI;
  uint8_t* SLO = sm + SM_SLO;
  uint8_t* KQ = sm + SM_KQ;
  uint8_t* KT = sm + SM_KT;
  uint8_t* RD = sm + SM_RD;
  uint8_t* TI = sm + SM_TI;
  uint8_t* XB = sm + SM_XB;
  float* OB = reinterpret_cast<float*>(sm + SM_RD);
  float* AB = reinterpret_cast<float*>(sm + SM_AB);
  uint8_t* ZB = sm + SM_ZB;
  float* g2_s = reinterpret_cast<float*>(sm + SM_VEC);   // chunk-local log2 decay
  float* G_s = g2_s + 64;
  float* b_s = G_s + 64;
  float* c_s = b_s + 64;
  float* la_s = c_s + 64;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + SM_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SM_BAR + 8);
  uint64_t* rbar = reinterpret_cast<uint64_t*>(sm + SM_BAR + 16);   // value / z row tiles

  const int tid = threadIdx.x, warp = tid >> 5;
  const int h = blockIdx.x;
  // Longest sequences first: block row y takes the sequence of rank y by
  // length (ties by index), so the long chains start in the first wave.
  int s = blockIdx.y;
  if (p.n_seq <= 256) {
    int* pick = reinterpret_cast<int*>(sm + SM_BAR + 12);
    if (tid == 0) *pick = blockIdx.y;
    __syncthreads();
    for (int q = tid; q < p.n_seq; q += PT) {
      const int lq = p.cu[q + 1] - p.cu[q];
      int rank = 0;
      for (int r = 0; r < p.n_seq; ++r) {
        const int lr = p.cu[r + 1] - p.cu[r];
        rank += (lr > lq) || (lr == lq && r < q);
      }
      if (rank == (int)blockIdx.y) *pick = q;
    }
    __syncthreads();
    s = *pick;
    __syncthreads();
  }
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
  const uint16_t* qkv = static_cast<const uint16_t*>(p.qkv);

  if (tid == 0) {
    tc::mbar_init(mbar, 1);
    tc::mbar_init(rbar, 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tslot, TM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tslot;
  const uint32_t lane_addr = tbase + ((uint32_t)(32 * (warp & 3)) << 16);
  const int i = tid & 127;                 // value row (TMEM lane) of this thread
  const bool owner = tid < 128;            // warps 0..3 own the rows; warps 4..7 help

  // ---- initial state: row i into TMEM (f32) and the bf16 hi/lo tiles
  float* Sg = p.state + (((int64_t)slot * Hv + h) * D) * D;
  const bool has_init = p.has_init[s] != 0;
  {
    const int cb0 = owner ? 0 : 4;                   // owners columns 0..63, helpers 64..127
#pragma unroll 1
    for (int cb = cb0; cb < cb0 + 4; ++cb) {
      float v[16];
      if (has_init) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 f = reinterpret_cast<const float4*>(Sg + (int64_t)i * D + 16 * cb)[q];
          v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
        }
      } else {
#pragma unroll
        for (int q = 0; q < 16; ++q) v[q] = 0.f;
      }
      tc::tmem_st16(lane_addr + TM_S + 16 * cb, v);
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        uint4 hi, lo;
        tc::split8(v + 8 * hlf, hi, lo);
        st16(SHI + tc::kmajor_offset(i, 16 * cb + 8 * hlf, 128), hi);
        st16(SLO + tc::kmajor_offset(i, 16 * cb + 8 * hlf, 128), lo);
      }
    }
    tc::tmem_st_wait();
  }

  uint32_t phase = 0, rphase = 0;
  bool timed_out = false;
  const uint32_t id128 = tc::idesc_bf16_f32(128, 128);
  const uint32_t id64 = tc::idesc_bf16_f32(128, 64);
  const uint32_t a_SHI = tc::smem_u32(SHI), a_SLO = tc::smem_u32(SLO), a_KQ = tc::smem_u32(KQ);
  const uint32_t a_KT = tc::smem_u32(KT), a_RD = tc::smem_u32(RD);
  const uint32_t a_XB = tc::smem_u32(XB);

  // Thread 0 commits the MMAs it issued; everyone waits (bounded). Returns
  // false, for the whole block, if the wait gave up.
  auto commit_and_wait = [&]() -> bool {
    if (tid == 0) tc::mma_commit(mbar);
    const bool ok = tc::mbar_wait(mbar, phase, WAIT_POLLS);
    if (ok) phase ^= 1;
    tc::fence_after_sync();
    return __syncthreads_or(!ok) == 0;
  };

  // Copies of a chunk's keys and queries (into the K-major [K;Q] tile, zero
  // past the sequence end) and raw gates, in flight while the previous chunk
  // finishes. Its value rows and the finished chunk's z rows come as one TMA
  // box each (64 rows x 128 columns) on the row barrier; rows past the sequence
  // end hold other tokens (zeros past n_tok) and are never used.
  float* al_raw = la_s;                                  // raw alpha until log2 is taken
  auto copy_rows = [&](bool v, int64_t vc0, bool zz, int64_t zc0) {
    if (tid == 0) {
      tc::fence_async_smem();                            // earlier reads of TI / ZB come first
      tc::mbar_arrive_expect_tx(rbar, (v ? 16384u : 0u) + (zz ? 16384u : 0u));
      if (v) tma_rows(TI, &vmap, (2 * Hk + h) * D, (int)vc0, rbar);
      if (zz) tma_rows(ZB, &zmap, h * D, (int)zc0, rbar);
    }
  };
  auto prefetch = [&](int64_t pc0, int pm) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {                        // keys / queries: a warp = 32 tokens
      const int it = tid + k * PT, t = it & 63, part = it >> 6, isq = part >> 4, w8 = part & 15;
      const int tt = t < pm ? t : 0;
      cp_async16(KQ + tc::kmajor_offset(isq * 64 + t, 8 * w8, 128),
                 qkv + (pc0 + tt) * C + (isq ? hq : Hk + hq) * D + 8 * w8, t < pm ? 16u : 0u);
    }
    if (tid < C64) {
      const int t = tid, tt = t < pm ? t : 0;
      const int64_t gi = (pc0 + tt) * Hv + h;
      if (p.gate_bf16) {                                 // 2-byte gates: plain loads
        al_raw[t] = t < pm ? load_gate(p.alpha, gi, 1) : 0.f;
        b_s[t] = t < pm ? load_gate(p.beta, gi, 1) : 0.f;
      } else {
        cp_async4(al_raw + t, static_cast<const float*>(p.alpha) + gi, t < pm ? 4u : 0u);
        cp_async4(b_s + t, static_cast<const float*>(p.beta) + gi, t < pm ? 4u : 0u);
      }
    }
    cp_async_commit();
  };

  // z-gated RMSNorm of a chunk's outputs by the 128 owner threads (16 lanes per
  // token, 8 tokens at a time). It runs while the helpers solve for the next
  // chunk's deltas: it reads only the output buffer and the staged z rows.
  auto epilogue = [&](int64_t ec0, int em) {
      const int l16 = tid & 15, lane = tid & 31;
      float nw[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) nw[j] = p.norm_w[l16 * 8 + j];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float zv[4][8], o[4][8], ss[4];
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int t = (4 * half + it) * 8 + (tid >> 4);
          load8<BF16>(ZB, (int64_t)t * D + l16 * 8, zv[it]);
          const float4 u0 = reinterpret_cast<const float4*>(OB + t * D)[2 * l16];
          const float4 u1 = reinterpret_cast<const float4*>(OB + t * D)[2 * l16 + 1];
          o[it][0] = u0.x; o[it][1] = u0.y; o[it][2] = u0.z; o[it][3] = u0.w;
          o[it][4] = u1.x; o[it][5] = u1.y; o[it][6] = u1.z; o[it][7] = u1.w;
          ss[it] = head_sum_sq16(o[it]);
        }
        // lanes with l16 % 4 == it take the 1/sqrt of token it (same bits as every lane)
        const int sel = l16 & 3;
        const float ssel = sel == 0 ? ss[0] : sel == 1 ? ss[1] : sel == 2 ? ss[2] : ss[3];
        const float rm = inv_norm(__fmul_rn(ssel, 1.0f / D), p.eps);
#pragma unroll
        for (int it = 0; it < 4; ++it) {
          const int t = (4 * half + it) * 8 + (tid >> 4);
          const float r = __shfl_sync(FULL, rm, (lane & ~3) | it);
          if (t < em) {
            float res[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
              res[j] = __fmul_rn(__fmul_rn(__fmul_rn(o[it][j], r), nw[j]), silu_gate(zv[it][j]));
            store_out8<BF16>(p.out, (ec0 + t) * Hv * D + (int64_t)h * D + l16 * 8, res, p.out_f32);
          }
        }
      }
  };

  int64_t prev_c0 = -1;
  int prev_m = 0;
  if (seq0 < seq1) {
    prefetch(seq0, (int)(seq1 - seq0 < C64 ? seq1 - seq0 : C64));
    copy_rows(true, seq0, false, 0);
  }
  for (int64_t c0 = seq0; c0 < seq1; c0 += C64) {
    const int m = (int)(seq1 - c0 < C64 ? seq1 - c0 : C64);

    // ---- (a) the prefetched chunk: wait for it, transpose the keys into K^T,
    //          take log2 of the gates (alpha = 1 past the end: zero-filled raw
    //          alpha is mapped to log2 = 0)
    cp_async_wait_all();
    {
      const bool ok = tc::mbar_wait(rbar, rphase, WAIT_POLLS);
      if (__syncthreads_or(!ok)) { timed_out = true; break; }
      rphase ^= 1;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {                        // key pieces: a warp = 32 tokens
      const int it = tid + k * PT, t = it & 63, w8 = it >> 6;
      const uint4 pc = *reinterpret_cast<const uint4*>(KQ + tc::kmajor_offset(t, 8 * w8, 128));
      const uint32_t wv[4] = {pc.x, pc.y, pc.z, pc.w};
#pragma unroll
      for (int u = 0; u < 8; ++u)
        *reinterpret_cast<uint16_t*>(KT + tc::kmajor_offset(8 * w8 + u, t, 128)) =
            (uint16_t)(wv[u >> 1] >> (16 * (u & 1)));
    }
    if (tid < C64) {
      float al = al_raw[tid];
      if (p.raw_gates) {                                 // raw projections: the gate step
        al = gate_alpha(al);                             // (tokens past the end keep beta = 0)
        if (tid < m) b_s[tid] = gate_beta(b_s[tid]);
      }
      la_s[tid] = tid < m ? log2f(al) : 0.f;
    }
    tc::fence_async_smem();
    __syncthreads();

    // ---- (b) MMA1 (S0 hi, lo) and MMA2, while warp 4 builds the decay tables
    //          (prefix sums of log2 alpha by a warp scan: lane l holds tokens 2l,
    //          2l + 1)
    if (tid == 0) {
      tc::fence_after_sync();
      mma_pass(tbase + TM_P, a_SHI, 128, a_KQ, 128, 8, id128, false);
      mma_pass(tbase + TM_P, a_SLO, 128, a_KQ, 128, 8, id128, true);
      mma_pass(tbase + TM_G, a_KQ, 128, a_KQ, 128, 8, id64, false);
    }
    if (warp == 4) {
      const int l = tid & 31;
      const float x0 = la_s[2 * l], x1 = la_s[2 * l + 1];
      float v = x0 + x1;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float n = __shfl_up_sync(FULL, v, off);
        if (l >= off) v += n;
      }
      float before = __shfl_up_sync(FULL, v, 1);        // sum of the tokens before 2l
      if (l == 0) before = 0.f;
      const float e0 = before + x0, e1 = e0 + x1;       // inclusive sums at 2l, 2l + 1
      g2_s[2 * l] = e0;
      g2_s[2 * l + 1] = e1;
      G_s[2 * l] = ex2(e0);
      G_s[2 * l + 1] = ex2(e1);
    }
    __syncthreads();
    if (tid < C64) c_s[tid] = ex2(g2_s[C64 - 1] - g2_s[tid]);
    if (!commit_and_wait()) { timed_out = true; break; }

    // ---- (c) tables from G (owners); R rows from P^T, kept in registers (helpers)
    float r[64];                                         // R, then d, of value row i (helpers)
    if (owner) {
      float gr[64];
#pragma unroll
      tc::tmem_ld16x4(lane_addr + TM_G, gr, lane_addr + TM_G + 16, gr + 16, lane_addr + TM_G + 32, gr + 32,
                      lane_addr + TM_G + 48, gr + 48);
      if (i < C64) {                                     // -A row i (f32, strictly lower), stored
        const float gi = g2_s[i], bi = b_s[i];           // as column i of -A^T
#pragma unroll
        for (int u = 0; u < C64; ++u)
          AB[u * AP + i] = u < i ? -__fmul_rn(__fmul_rn(bi, ex2(gi - g2_s[u])), gr[u]) : 0.f;
      } else {                                           // X row t: the MMA5 B tile
        const int t = i - C64;
        const float gt = g2_s[t];
        float x[64];
#pragma unroll
        for (int u = 0; u < C64; ++u) x[u] = u <= t ? __fmul_rn(ex2(gt - g2_s[u]), gr[u]) : 0.f;
        put_row64(XB, XB + 8192, t, 64, x);
      }
    } else {
      const uint16_t* vcol = reinterpret_cast<const uint16_t*>(TI) + i;   // staged values
#pragma unroll
      for (int cb = 0; cb < 4; cb += 2) {
        float pk[2][16];
        tc::tmem_ld16x2(lane_addr + TM_P + 16 * cb, pk[0], lane_addr + TM_P + 16 * cb + 16, pk[1]);
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int t = 16 * cb + u;
          const float vt = t < m ? bf2f(vcol[t * D]) : 0.f;   // rows past m: other tokens
          const float bt = b_s[t];
          r[t] = __fmaf_rn(-__fmul_rn(bt, G_s[t]), pk[u >> 4][u & 15], __fmul_rn(bt, vt));
        }
      }
    }
    __syncthreads();                                     // A complete

    // ---- (d) helpers: (I + A) d = R for value row i, in blocks of 16 tokens:
    //          block k first takes the updates d_t += (-A[t][s]) d_s of every
    //          finished token s < 16k in ascending s (a rolled loop reading d_s
    //          back from shared memory), then solves its diagonal block by
    //          right-looking substitution. Every d_t gets the same fused
    //          multiply-adds in the same order (ascending s) as a plain forward
    //          substitution; the rolled loop keeps the code small enough for the
    //          instruction cache. Column s of -A is read as float4s from -A^T.
    //          Owners: the previous chunk's z-gated RMSNorm
    if (owner) {
      if (prev_c0 >= 0) epilogue(prev_c0, prev_m);
    } else {
      float* DS = reinterpret_cast<float*>(KQ);          // d values [token][value row]; KQ is free
#pragma unroll
      for (int k = 0; k < 4; ++k) {
#pragma unroll 4
        for (int sv = 0; sv < 16 * k; ++sv) {
          const float ds = DS[sv * D + i];
          const float2 d2 = make_float2(ds, ds);
          const float4* acol = reinterpret_cast<const float4*>(AB + sv * AP) + 4 * k;
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            const float4 a = acol[j4];
            const int t = 16 * k + 4 * j4;
            const float2 lo = __ffma2_rn(make_float2(a.x, a.y), d2, make_float2(r[t], r[t + 1]));
            const float2 hi = __ffma2_rn(make_float2(a.z, a.w), d2, make_float2(r[t + 2], r[t + 3]));
            r[t] = lo.x; r[t + 1] = lo.y; r[t + 2] = hi.x; r[t + 3] = hi.y;
          }
        }
#pragma unroll
        for (int u = 16 * k; u < 16 * k + 15; ++u) {
          const float du = r[u];
          const float* acol = AB + u * AP;
#pragma unroll
          for (int t = u + 1; t < 16 * k + 16; ++t) r[t] = __fmaf_rn(acol[t], du, r[t]);
        }
        if (k < 3) {
#pragma unroll
          for (int j = 0; j < 16; ++j) DS[(16 * k + j) * D + i] = r[16 * k + j];
        }
      }
    }
    __syncthreads();                                     // the output buffer has been read

    // ---- (f) helpers: D^T row i -> MMA5 A tile, (c D)^T row i -> MMA3 A tile
    if (!owner) {
      put_row64(RD, RD + 16384, i, 128, r);
#pragma unroll
      for (int u = 0; u < C64; ++u) r[u] = __fmul_rn(c_s[u], r[u]);
      put_row64(KQ, KQ + 16384, i, 128, r);
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();

    // ---- (g) MMA5: O^T = D^T X^T;  MMA3: dS = (c D)^T K
    if (tid == 0) {
      tc::fence_after_sync();
      mma_pass(tbase + TM_O, a_RD, 128, a_XB, 64, 4, id64, false);
      mma_pass(tbase + TM_O, a_RD + 16384, 128, a_XB, 64, 4, id64, true);
      mma_pass(tbase + TM_O, a_RD, 128, a_XB + 8192, 64, 4, id64, true);
      mma_pass(tbase + TM_DS, a_KQ, 128, a_KT, 128, 4, id128, false);
      mma_pass(tbase + TM_DS, a_KQ + 16384, 128, a_KT, 128, 4, id128, true);
    }
    if (!commit_and_wait()) { timed_out = true; break; }

    if (c0 + C64 < seq1) {                               // next chunk's inputs: KQ and TI are free
      const int64_t n0 = c0 + C64;
      prefetch(n0, (int)(seq1 - n0 < C64 ? seq1 - n0 : C64));
      copy_rows(true, n0, true, c0);                     // and this chunk's z rows
    } else {
      copy_rows(false, 0, true, c0);
    }

    // ---- (h) owners: o = G (S0 q) + O^T into the output buffer (the RD region
    //          is free now); helpers: S = G_last S + dS, TMEM and hi/lo tiles
    if (owner) {
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        float pq[16], ov[16];
        tc::tmem_ld16x2(lane_addr + TM_P + 64 + 16 * cb, pq, lane_addr + TM_O + 16 * cb, ov);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int t = 16 * cb + u;
          OB[t * D + i] = __fmul_rn(__fmaf_rn(G_s[t], pq[u], ov[u]), p.q_scale);
        }
      }
    } else {
      const float gl = G_s[C64 - 1];
#pragma unroll 1
      for (int cb0 = 0; cb0 < 8; cb0 += 2) {             // two 16-column blocks per TMEM wait
        float sv[2][16], dv[2][16];
        tc::tmem_ld16x4(lane_addr + TM_S + 16 * cb0, sv[0], lane_addr + TM_DS + 16 * cb0, dv[0],
                        lane_addr + TM_S + 16 * cb0 + 16, sv[1], lane_addr + TM_DS + 16 * cb0 + 16, dv[1]);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int cb = cb0 + k;
#pragma unroll
          for (int u = 0; u < 16; ++u) sv[k][u] = __fmaf_rn(gl, sv[k][u], dv[k][u]);
          tc::tmem_st16(lane_addr + TM_S + 16 * cb, sv[k]);
#pragma unroll
          for (int hlf = 0; hlf < 2; ++hlf) {
            uint4 hi, lo;
            tc::split8(sv[k] + 8 * hlf, hi, lo);
            st16(SHI + tc::kmajor_offset(i, 16 * cb + 8 * hlf, 128), hi);
            st16(SLO + tc::kmajor_offset(i, 16 * cb + 8 * hlf, 128), lo);
          }
        }
      }
      tc::tmem_st_wait();
    }
    tc::fence_before_sync();
    __syncthreads();
    prev_c0 = c0;
    prev_m = m;
  }
  if (!timed_out && prev_c0 >= 0) {                     // the last chunk
    const bool ok = tc::mbar_wait(rbar, rphase, WAIT_POLLS);
    if (__syncthreads_or(!ok)) timed_out = true;
    else {
      rphase ^= 1;
      if (owner) epilogue(prev_c0, prev_m);
    }
  }

  if (timed_out) {
    if (tid == 0) report(p.dev_err, GDN_DEVERR_TIMEOUT);
    tc::mbar_wait(mbar, phase, WAIT_POLLS);              // the pending phase: work in flight
    tc::mbar_wait(rbar, rphase, WAIT_POLLS);             // row tiles in flight
    cp_async_wait_all();
  } else {
    const int cb0 = owner ? 0 : 4;                       // final state: row i from TMEM
#pragma unroll 1
    for (int cb = cb0; cb < cb0 + 4; ++cb) {
      float v[16];
      tc::tmem_ld16(lane_addr + TM_S + 16 * cb, v);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        reinterpret_cast<float4*>(Sg + (int64_t)i * D + 16 * cb)[q] =
            make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tbase, TM_COLS);
}

size_t prefill_tc_smem_bytes() { return SM_TOTAL; }

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t stream) {
  const int smem = (int)SM_TOTAL;
  cudaError_t e = set_smem_once<prefill_tc_kernel>(smem);
  if (e != cudaSuccess) return e;
  CUtensorMap vmap, zmap;
  const uint64_t C = (uint64_t)(2 * a.Hk + a.Hv) * D;
  e = encode_bf16_rows_map(&vmap, a.qkv, (uint64_t)a.n_tok, C, C, D, C64);
  if (e != cudaSuccess) return e;
  e = encode_bf16_rows_map(&zmap, a.z, (uint64_t)a.n_tok, (uint64_t)a.Hv * D, (uint64_t)a.Hv * D, D, C64);
  if (e != cudaSuccess) return e;
  dim3 grid(a.Hv, a.n_seq);
  prefill_tc_kernel<<<grid, PT, smem, stream>>>(a, vmap, zmap);
  return cudaGetLastError();
}

}  // namespace gdn
