// Causal conv1d (width 4) + SiLU (+ q/k L2 norm) over varlen sequences in exact
// 64-token chunks, and the standalone post-conv L2 norm.
//
// Source: "perf(gdn): optimize post-conv and causal-conv kernels - #155"
// ("Blocker": the width-4 causal conv over c channels; "Merged ...": the 128-lane
// sum of squares then 1/sqrtf; "New issue #305": only the chunk-0 block reads
// the initial conv_state while the last chunk wrote the final one — a race).
//
// Design (GB300): one thread owns 8 contiguous channels (one 16-byte bf16 load)
// and walks the 64 tokens of its chunk, keeping the 3 previous rows in
// registers, so x is read once (plus a 3-row halo per chunk, an L2 hit). A warp
// holds two heads x 16 lanes, which is exactly the lane layout of the fixed
// sum-of-squares tree. The chunk-0 thread that reads a channel's initial rows
// is the one that later writes that channel's final rows: the final rows are
// taken from x (or from the initial rows it holds when the sequence is shorter
// than 3), so no other block ever touches conv_state.
#include "common.cuh"
#include "launch.h"

namespace gdn {

constexpr int CONV_THREADS = 256;
constexpr int CONV_QUARTERS = 4;                      // token quarters of a chunk
constexpr int CONV_TOK = CHUNK / CONV_QUARTERS;       // 16 tokens per thread
constexpr int CONV_HEADS_PER_BLOCK = 4;               // 4 heads x 16 lanes x 4 quarters
constexpr int CONV_BATCH = 2;                         // tokens loaded ahead per step

// Thread layout: warp w covers quarter w / 2 of the chunk and heads
// 2 (w % 2), 2 (w % 2) + 1 of the block's 4 heads (16 lanes each, 8 contiguous
// channels per lane). Quarter 0 of the chunk-0 block owns conv_state.
template <int A, bool NORM>
__global__ void __launch_bounds__(CONV_THREADS, 2)
conv_fwd_kernel(const void* __restrict__ x, int64_t ld_x, void* __restrict__ y, int64_t ld_y,
                const void* __restrict__ conv_w, void* __restrict__ conv_state,
                const int32_t* __restrict__ slot_idx, const int32_t* __restrict__ cu,
                const uint8_t* __restrict__ has_init, int n_seq, int64_t n_tok, int n_heads,
                int n_qk, int n_slots, float eps, uint32_t* dev_err) {
  int s, ci;
  if (!find_chunk(cu, n_seq, blockIdx.x, CHUNK, s, ci)) return;
  const int slot = slot_idx[s];
  if (slot < 0) return;                                  // padding sequence
  const int64_t seq0 = cu[s], seq1 = cu[s + 1];
  if (seq1 < seq0 || seq0 < 0 || seq1 > n_tok) {
    if (ci == 0 && threadIdx.x == 0 && blockIdx.y == 0) report(dev_err, GDN_DEVERR_SEQLENS);
    return;
  }
  if (slot >= n_slots) {
    if (ci == 0 && threadIdx.x == 0 && blockIdx.y == 0) report(dev_err, GDN_DEVERR_SLOT);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp >> 1;
  const int head = blockIdx.y * CONV_HEADS_PER_BLOCK + (warp & 1) * 2 + (lane >> 4);
  const bool active = head < n_heads;                    // uniform per 16 lanes
  const bool is_qk = head < 2 * n_qk;
  const int C = n_heads * D;
  const int c0 = head * D + (lane & 15) * 8;
  const int64_t len = seq1 - seq0;
  const int64_t t_chunk = seq0 + (int64_t)ci * CHUNK;
  const int64_t t_end = min(t_chunk + CHUNK, seq1);
  const int64_t t_begin = t_chunk + quarter * CONV_TOK;    // this thread's tokens
  const int64_t t_stop = min(t_begin + CONV_TOK, t_end);
  const bool owner = ci == 0 && quarter == 0;             // reads and writes conv_state
  const int64_t st_base = (int64_t)slot * KS * C;

  if (t_begin < t_stop) {                                 // uniform per warp
    float2 w[4][4];                                       // [channel pair][tap]
    float2 p0[4], p1[4], p2[4];                           // the three previous rows
    if (active) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {                      // channels 2q, 2q+1: 8 taps
        float t8[8];
        load8<A>(conv_w, (int64_t)c0 * KW + 8 * q, t8);
#pragma unroll
        for (int j = 0; j < 4; ++j) w[q][j] = make_float2(t8[j], t8[4 + j]);
      }
      float r0[8], r1[8], r2[8];
      if (owner) {
        if (has_init[s]) {
          load8<A>(conv_state, st_base + c0, r0);
          load8<A>(conv_state, st_base + C + c0, r1);
          load8<A>(conv_state, st_base + 2 * (int64_t)C + c0, r2);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) { r0[j] = 0.f; r1[j] = 0.f; r2[j] = 0.f; }
        }
      } else {
        load8<A>(x, (t_begin - 3) * ld_x + c0, r0);
        load8<A>(x, (t_begin - 2) * ld_x + c0, r1);
        load8<A>(x, (t_begin - 1) * ld_x + c0, r2);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        p0[q] = make_float2(r0[2 * q], r0[2 * q + 1]);
        p1[q] = make_float2(r1[2 * q], r1[2 * q + 1]);
        p2[q] = make_float2(r2[2 * q], r2[2 * q + 1]);
      }
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        p0[q] = p1[q] = p2[q] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 4; ++j) w[q][j] = make_float2(0.f, 0.f);
      }
    }

    // 16 tokens, fully unrolled so the three-row window rotates through
    // registers. Rows stay packed until used, and the loads of the next batch
    // of CONV_BATCH tokens are issued before the current batch is computed.
    const int n_here = (int)(t_stop - t_begin);           // 1..16, uniform per warp
    Raw8<A> cur[CONV_BATCH], nxt[CONV_BATCH];
#pragma unroll
    for (int u = 0; u < CONV_BATCH; ++u) {
      if (active && u < n_here) raw_load<A>(x, (t_begin + u) * ld_x + c0, cur[u]);
      else raw_zero<A>(cur[u]);
    }
#pragma unroll
    for (int b0 = 0; b0 < CONV_TOK; b0 += CONV_BATCH) {
      if (b0 >= n_here) break;
      if (b0 + CONV_BATCH < CONV_TOK) {
#pragma unroll
        for (int u = 0; u < CONV_BATCH; ++u) {
          const int tt = b0 + CONV_BATCH + u;
          if (active && tt < n_here) raw_load<A>(x, (t_begin + tt) * ld_x + c0, nxt[u]);
          else raw_zero<A>(nxt[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < CONV_BATCH; ++u) {
        if (b0 + u >= n_here) break;
        float xv[8], v[8];
        raw_unpack<A>(cur[u], xv);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 cv = make_float2(xv[2 * q], xv[2 * q + 1]);
          const float2 a = silu2(conv4x2(w[q][0], w[q][1], w[q][2], w[q][3], p0[q], p1[q], p2[q], cv));
          v[2 * q] = a.x;
          v[2 * q + 1] = a.y;
          p0[q] = p1[q]; p1[q] = p2[q]; p2[q] = cv;
        }
        if constexpr (NORM) {
          const float ss = head_sum_sq16(v);           // all lanes take part
          if (is_qk) {
            const float r = inv_norm(ss, eps);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float2 o = __fmul2_rn(make_float2(v[2 * q], v[2 * q + 1]), make_float2(r, r));
              v[2 * q] = o.x;
              v[2 * q + 1] = o.y;
            }
          }
        }
        if (active) store8<A>(y, (t_begin + b0 + u) * ld_y + c0, v);
      }
#pragma unroll
      for (int u = 0; u < CONV_BATCH; ++u) cur[u] = nxt[u];
    }
  }

  // Final conv_state: rows len, len+1, len+2 of (initial rows ++ x rows),
  // written by the thread that read the initial rows, after its last read.
  // When len < 3 new row r is old row len + r >= r; rows are rewritten in
  // ascending order, so each old row is read before it is overwritten.
  if (owner && active) {
    const bool hi = has_init[s] != 0;
#pragma unroll
    for (int r = 0; r < 3; ++r) {
      const int64_t idx = len + r;
      float v[8];
      if (idx >= 3) load8<A>(x, (seq0 + idx - 3) * ld_x + c0, v);
      else if (hi) load8<A>(conv_state, st_base + idx * C + c0, v);
      else {
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = 0.f;
      }
      store8<A>(conv_state, st_base + (int64_t)r * C + c0, v);
    }
  }
}

// Standalone per-head L2 norm of q and k heads; v channels copied.
template <int AI, int AO>
__global__ void __launch_bounds__(256)
postconv_norm_kernel(const void* __restrict__ yin, void* __restrict__ yout, int64_t n_tok,
                     int n_heads, int n_qk, float eps) {
  const int64_t groups = n_tok * n_heads;                 // (token, head) pairs
  const int lane16 = threadIdx.x & 15;
  // 16 lanes per (token, head); grid-stride over pairs in steps that keep the
  // 16-lane groups aligned inside warps.
  const int64_t stride = (int64_t)gridDim.x * (blockDim.x / 16);
  for (int64_t g = (int64_t)blockIdx.x * (blockDim.x / 16) + (threadIdx.x >> 4);
       g - ((threadIdx.x >> 4) & 1) < groups; g += stride) {
    const bool live = g < groups;
    const int64_t tok = live ? g / n_heads : 0;
    const int head = live ? int(g % n_heads) : 0;
    const int64_t e0 = tok * (int64_t)n_heads * D + head * D + lane16 * 8;
    float v[8];
    if (live) load8<AI>(yin, e0, v);
    else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = 0.f;
    }
    const float ss = head_sum_sq16(v);                    // all 32 lanes take part
    if (live && head < 2 * n_qk) {
      const float r = inv_norm(ss, eps);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = __fmul_rn(v[j], r);
    }
    if (live) store8<AO>(yout, e0, v);
  }
}

// ------------------------------------------------------------------ launchers
cudaError_t launch_conv_fwd(const gdn_config& cfg, const void* x, int64_t ld_x, void* y,
                            int64_t ld_y, const void* conv_w, void* conv_state,
                            const int32_t* slot_idx, const int32_t* cu, const uint8_t* has_init,
                            int n_seq, int64_t n_tok, int fuse_norm, cudaStream_t stream) {
  const int n_heads = 2 * cfg.n_qk_heads + cfg.n_v_heads;
  const int64_t max_chunks = (n_tok + CHUNK - 1) / CHUNK + n_seq;
  dim3 grid((unsigned)max_chunks, (n_heads + CONV_HEADS_PER_BLOCK - 1) / CONV_HEADS_PER_BLOCK);
#define GDN_CONV_ARGS                                                                     \
  x, ld_x, y, ld_y, conv_w, conv_state, slot_idx, cu, has_init, n_seq, n_tok, n_heads,   \
      cfg.n_qk_heads, cfg.n_slots, cfg.eps, cfg.dev_err
  if (cfg.act == GDN_BF16) {
    if (fuse_norm) conv_fwd_kernel<BF16, true><<<grid, CONV_THREADS, 0, stream>>>(GDN_CONV_ARGS);
    else conv_fwd_kernel<BF16, false><<<grid, CONV_THREADS, 0, stream>>>(GDN_CONV_ARGS);
  } else {
    if (fuse_norm) conv_fwd_kernel<F32, true><<<grid, CONV_THREADS, 0, stream>>>(GDN_CONV_ARGS);
    else conv_fwd_kernel<F32, false><<<grid, CONV_THREADS, 0, stream>>>(GDN_CONV_ARGS);
  }
#undef GDN_CONV_ARGS
  return cudaGetLastError();
}

cudaError_t launch_postconv_norm(const gdn_config& cfg, int in_t, const void* yin, int out_t,
                                 void* yout, int64_t n_tok, int n_sm, cudaStream_t stream) {
  const int n_heads = 2 * cfg.n_qk_heads + cfg.n_v_heads;
  const int64_t groups = n_tok * n_heads;
  const int per_block = 256 / 16;
  int64_t blocks = (groups + per_block - 1) / per_block;
  const int64_t cap = (int64_t)n_sm * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  dim3 grid((unsigned)blocks);
#define GDN_PCN_ARGS yin, yout, n_tok, n_heads, cfg.n_qk_heads, cfg.eps
  if (in_t == GDN_F32 && out_t == GDN_F32) postconv_norm_kernel<F32, F32><<<grid, 256, 0, stream>>>(GDN_PCN_ARGS);
  else if (in_t == GDN_F32) postconv_norm_kernel<F32, BF16><<<grid, 256, 0, stream>>>(GDN_PCN_ARGS);
  else if (out_t == GDN_F32) postconv_norm_kernel<BF16, F32><<<grid, 256, 0, stream>>>(GDN_PCN_ARGS);
  else postconv_norm_kernel<BF16, BF16><<<grid, 256, 0, stream>>>(GDN_PCN_ARGS);
#undef GDN_PCN_ARGS
  return cudaGetLastError();
}

}  // namespace gdn
