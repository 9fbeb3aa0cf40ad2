// Causal conv1d (width 4) + SiLU (+ q/k L2 norm) over varlen sequences in exact
// 64-token chunks, and the standalone post-conv L2 norm.
//
// Source: "perf(gdn): optimize post-conv and causal-conv kernels - #155"
// ("Blocker": the width-4 causal conv over c channels; "Merged ...": the 128-lane
// sum of squares then 1/sqrtf; "New issue #305": only the chunk-0 block reads
// the initial conv_state while the last chunk wrote the final one — a race).
//
// Design (GB300). A block takes one 64-token chunk of one sequence and four
// heads. Warp 0 bulk-copies (TMA) the chunk's rows of those heads, with the 3
// rows before it (the initial conv_state rows for chunk 0), into shared memory
// at once, all counted on one mbarrier, so a whole 67 KiB tile is in flight per
// block. One thread then owns 8 contiguous channels of a quarter of the chunk
// (16 tokens) and walks them with the 3 previous rows in registers. A warp holds
// two heads x 16 lanes, which is exactly the lane layout of the fixed
// sum-of-squares tree; tokens go in pairs so that even lanes take the 1/sqrt of
// the first token and odd lanes of the second. The chunk-0 thread that reads a
// channel's initial rows is the one that later writes that channel's final
// rows: the final rows are taken from x (or from the initial rows when the
// sequence is shorter than 3), so no other block ever touches conv_state.
#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace gdn {

constexpr int CONV_HEADS_PER_BLOCK = 4;               // 4 heads x 16 lanes x 4 quarters
constexpr int CONV_QUARTERS = 4;                      // token quarters of a chunk
constexpr int CONV_THREADS = CONV_HEADS_PER_BLOCK * 16 * CONV_QUARTERS;
constexpr int CONV_TOK = CHUNK / CONV_QUARTERS;       // 16 tokens per thread
constexpr int CONV_ROWS = KS + CHUNK;                 // staged rows: 3 before the chunk + 64

template <int A> constexpr int conv_tile_bytes() { return CONV_ROWS * CONV_HEADS_PER_BLOCK * D * (A == BF16 ? 2 : 4); }

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
  extern __shared__ __align__(128) uint8_t tile[];      // [CONV_ROWS][4 heads x 128] act
  __shared__ uint64_t bar;
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
  constexpr int asz = A == BF16 ? 2 : 4;
  constexpr int ROW = CONV_HEADS_PER_BLOCK * D;           // tile row stride in elements
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int head0 = blockIdx.y * CONV_HEADS_PER_BLOCK;
  const int heads_here = min(CONV_HEADS_PER_BLOCK, n_heads - head0);
  const int C = n_heads * D;
  const int64_t len = seq1 - seq0;
  const int64_t t_chunk = seq0 + (int64_t)ci * CHUNK;
  const int n_here = (int)(min(t_chunk + CHUNK, seq1) - t_chunk);   // 0 only for an empty sequence
  const bool hi = has_init[s] != 0;
  const int64_t st_base = (int64_t)slot * KS * C;

  // ---- stage rows t_chunk - 3 .. t_chunk + n_here - 1 (tile row r = token t_chunk - 3 + r)
  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  __syncthreads();                                       // the barrier is initialised before any wait
  const bool halo_x = ci > 0, halo_state = ci == 0 && hi;
  if (warp == 0) {
    const uint32_t row_bytes = (uint32_t)heads_here * D * asz;
    if (lane == 0)
      tc::mbar_arrive_expect_tx(&bar, (uint32_t)(n_here + ((halo_x || halo_state) ? KS : 0)) * row_bytes);
    __syncwarp();
    for (int r = lane; r < KS + n_here; r += 32) {
      const char* src = nullptr;
      if (r >= KS || halo_x)
        src = static_cast<const char*>(x) + ((t_chunk - KS + r) * ld_x + (int64_t)head0 * D) * asz;
      else if (halo_state)
        src = static_cast<const char*>(conv_state) + (st_base + (int64_t)r * C + (int64_t)head0 * D) * asz;
      if (src) tc::bulk_load(tile + (size_t)r * ROW * asz, src, row_bytes, &bar);
    }
  }
  if (!halo_x && !halo_state) {                          // chunk 0 without initial rows: zeros
    for (int e = tid; e < KS * ROW * asz / 16; e += CONV_THREADS)
      reinterpret_cast<uint4*>(tile)[e] = make_uint4(0u, 0u, 0u, 0u);
  }
  const int quarter = warp >> 1;
  const int hb = (warp & 1) * 2 + (lane >> 4);           // head within the block
  const int head = head0 + hb;
  const bool active = hb < heads_here;                   // uniform per 16 lanes
  const bool is_qk = head < 2 * n_qk;
  const int c0 = head * D + (lane & 15) * 8;             // global channel
  const int cb = hb * D + (lane & 15) * 8;               // channel within a tile row
  const int u0 = quarter * CONV_TOK;                     // this thread's first token in the chunk
  const int n_mine = max(0, min(CONV_TOK, n_here - u0)); // uniform per warp
  const bool owner = ci == 0 && quarter == 0;            // reads and writes conv_state
  Raw8<A> wr[4];                                          // the taps, in flight with the tile
  if (active && n_mine > 0) {
#pragma unroll
    for (int q = 0; q < 4; ++q) raw_load<A>(conv_w, (int64_t)c0 * KW + 8 * q, wr[q]);
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) raw_zero<A>(wr[q]);
  }
  const bool ok = tc::mbar_wait(&bar, 0, 1u << 24);
  if (__syncthreads_or(!ok)) {                           // also orders the zero rows
    if (tid == 0) report(dev_err, GDN_DEVERR_TIMEOUT);
    tc::mbar_wait(&bar, 0, 1u << 24);                    // the copies, if still in flight
    return;
  }

  if (n_mine > 0) {
    float2 w[4][4];                                       // [channel pair][tap]
    float2 p0[4], p1[4], p2[4];                           // the three previous rows
    {
      float r0[8], r1[8], r2[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {                      // channels 2q, 2q+1: 8 taps
        float t8[8];
        raw_unpack<A>(wr[q], t8);
#pragma unroll
        for (int j = 0; j < 4; ++j) w[q][j] = make_float2(t8[j], t8[4 + j]);
      }
      load8<A>(tile, (int64_t)u0 * ROW + cb, r0);        // tile rows u0 .. u0 + 2 = tokens u0 - 3 ..
      load8<A>(tile, (int64_t)(u0 + 1) * ROW + cb, r1);
      load8<A>(tile, (int64_t)(u0 + 2) * ROW + cb, r2);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        p0[q] = make_float2(r0[2 * q], r0[2 * q + 1]);
        p1[q] = make_float2(r1[2 * q], r1[2 * q + 1]);
        p2[q] = make_float2(r2[2 * q], r2[2 * q + 1]);
      }
    }
    // 16 tokens in pairs, fully unrolled so the three-row window rotates through
    // registers. A pair's second token may lie past the chunk's end: its tile
    // row was not staged and its values are discarded.
#pragma unroll
    for (int u = 0; u < CONV_TOK; u += 2) {
      if (u >= n_mine) break;                             // uniform per warp
      float v[2][8];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        float xv[8];
        load8<A>(tile, (int64_t)(u0 + u + k + KS) * ROW + cb, xv);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 cv = make_float2(xv[2 * q], xv[2 * q + 1]);
          const float2 a = silu2(conv4x2(w[q][0], w[q][1], w[q][2], w[q][3], p0[q], p1[q], p2[q], cv));
          v[k][2 * q] = a.x;
          v[k][2 * q + 1] = a.y;
          p0[q] = p1[q]; p1[q] = p2[q]; p2[q] = cv;
        }
      }
      if constexpr (NORM) {
        const float ss0 = head_sum_sq16(v[0]);            // all lanes take part
        const float ss1 = head_sum_sq16(v[1]);
        const float rm = inv_norm((lane & 1) ? ss1 : ss0, eps);   // even lanes token u, odd u + 1
        const float r0 = __shfl_sync(FULL, rm, lane & ~1);
        const float r1 = __shfl_sync(FULL, rm, lane | 1);
        if (is_qk) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 o0 = __fmul2_rn(make_float2(v[0][2 * q], v[0][2 * q + 1]), make_float2(r0, r0));
            const float2 o1 = __fmul2_rn(make_float2(v[1][2 * q], v[1][2 * q + 1]), make_float2(r1, r1));
            v[0][2 * q] = o0.x; v[0][2 * q + 1] = o0.y;
            v[1][2 * q] = o1.x; v[1][2 * q + 1] = o1.y;
          }
        }
      }
      if (active) {
        store8<A>(y, (t_chunk + u0 + u) * ld_y + c0, v[0]);
        if (u + 1 < n_mine) store8<A>(y, (t_chunk + u0 + u + 1) * ld_y + c0, v[1]);
      }
    }
  }

  // Final conv_state: rows len, len+1, len+2 of (initial rows ++ x rows),
  // written by the thread that read the initial rows, after its last read.
  // When len < 3 new row r is old row len + r >= r; rows are rewritten in
  // ascending order, so each old row is read before it is overwritten.
  if (owner && active) {
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
template <int A, bool NORM, typename... Args>
static cudaError_t launch_conv_variant(dim3 grid, cudaStream_t stream, Args... args) {
  const int smem = conv_tile_bytes<A>();
  cudaError_t e = set_smem_once<conv_fwd_kernel<A, NORM>>(smem);
  if (e != cudaSuccess) return e;
  conv_fwd_kernel<A, NORM><<<grid, CONV_THREADS, smem, stream>>>(args...);
  return cudaSuccess;
}

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
  cudaError_t e;
  if (cfg.act == GDN_BF16) {
    e = fuse_norm ? launch_conv_variant<BF16, true>(grid, stream, GDN_CONV_ARGS)
                  : launch_conv_variant<BF16, false>(grid, stream, GDN_CONV_ARGS);
  } else {
    e = fuse_norm ? launch_conv_variant<F32, true>(grid, stream, GDN_CONV_ARGS)
                  : launch_conv_variant<F32, false>(grid, stream, GDN_CONV_ARGS);
  }
#undef GDN_CONV_ARGS
  if (e != cudaSuccess) return e;
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
