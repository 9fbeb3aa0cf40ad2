// Causal conv1d (width 4) + SiLU (+ q/k L2 norm) over varlen sequences in exact
// 64-token chunks, and the standalone post-conv L2 norm.
//
// Source: "perf(gdn): optimize post-conv and causal-conv kernels - #155"
// ("Blocker": the width-4 causal conv over c channels; "Merged ...": the 128-lane
// sum of squares then 1/sqrtf; "New issue #305": only the chunk-0 block reads
// the initial conv_state while the last chunk wrote the final one — a race).
//
// Design (GB300). The work items are (64-token chunk of one sequence, group
// of four heads). A persistent grid of one 512-thread block per SM walks them
// round-robin; each block keeps three tile buffers in shared memory and has the
// tiles of its next two items in flight (bulk copies, TMA) while it computes the
// current one, so HBM streams while the SM computes. A tile is the chunk's rows
// of its four heads with the 3 rows before it (x rows, or the initial conv_state
// rows for chunk 0), kept as two halves of two heads each, [67 rows][256
// channels]: the 64 chunk rows of a half arrive as one 2-D TMA box (256 x 64),
// the 3 rows before it as three row copies. One thread owns 8 contiguous
// channels of an eighth of the chunk (8 tokens) and walks them with the 3
// previous rows in registers. A warp holds two heads x 16 lanes, which is
// exactly the lane layout of the fixed sum-of-squares tree; the eight token sums
// of a head are reduced across its 16 lanes by halving exchanges (each lane ends
// with one token's sum, the per-token tree's bits), so one 1/sqrt per lane serves
// the eight tokens. A warp releases its tile stage once its conv loop has read
// it, before the norms and stores. The chunk-0 thread that reads a channel's
// initial rows is the one that later writes that channel's final rows: the
// final rows are taken from x (or from the initial rows when the sequence is
// shorter than 3), so no other block ever touches conv_state.
#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace gdn {

constexpr int CONV_HEADS_PER_BLOCK = 4;               // 4 heads x 16 lanes x 8 token groups
constexpr int CONV_GROUPS = 8;                        // token groups of a chunk
constexpr int CONV_THREADS = CONV_HEADS_PER_BLOCK * 16 * CONV_GROUPS;
constexpr int CONV_TOK = CHUNK / CONV_GROUPS;         // 8 tokens per thread
constexpr int CONV_ROWS = KS + CHUNK;                 // staged rows: 3 before the chunk + 64

constexpr int CONV_HALF_COLS = 2 * D;                 // two heads per TMA box
template <int A> __host__ __device__ constexpr int conv_half_bytes() { return CONV_ROWS * CONV_HALF_COLS * (A == BF16 ? 2 : 4); }
// The item's conv_w rows ([4 heads x 128 channels][4 taps]) follow the two halves.
template <int A> __host__ __device__ constexpr int conv_w_bytes() { return CONV_HEADS_PER_BLOCK * D * KW * (A == BF16 ? 2 : 4); }
template <int A> __host__ __device__ constexpr int conv_tile_bytes() { return 2 * conv_half_bytes<A>() + conv_w_bytes<A>(); }
// Tile buffers: three for bf16 (213 KiB), one for f32 (142 KiB; the f32 path is
// the test arm, not a streaming workload).
template <int A> __host__ __device__ constexpr int conv_stages() { return A == BF16 ? 3 : 1; }

// What a block knows about a staged item (written by the issuing thread before
// its arrival on the stage's barrier, read after the wait).
struct ConvItem {
  int s, ci, head0, flags;                               // flags: CI_*
  int slot, n_here;                                      // the sequence's slot, tokens in the chunk
  int64_t t_chunk, seq0, len;                            // first token row, sequence start and length
};
constexpr int CI_VALID = 1, CI_HALO_X = 2, CI_HALO_STATE = 4, CI_BAD_SLOT = 8, CI_BAD_SEQ = 16;

// 2-D TMA copy of a box of the x rows (x = column, y = row), counted on `bar`.
__device__ __forceinline__ void tma_box(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          tc::smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(tc::smem_u32(bar))
      : "memory");
}

// Thread layout: warp w covers token group w / 2 of the chunk (tokens 8 (w / 2)
// .. + 7) and heads 2 (w % 2), 2 (w % 2) + 1 of the item's 4 heads (16 lanes
// each, 8 contiguous channels per lane), which are tile half w % 2. Group 0 of
// the chunk-0 item owns conv_state. xmap: x as [n_tok rows][C columns] in boxes
// of 256 columns x 64 rows (rows past n_tok and columns past C read as zeros).
template <int A, bool NORM>
__global__ void __launch_bounds__(CONV_THREADS, 1)
conv_fwd_kernel(const void* __restrict__ x, int64_t ld_x, void* __restrict__ y, int64_t ld_y,
                const void* __restrict__ conv_w, void* __restrict__ conv_state,
                const int32_t* __restrict__ slot_idx, const int32_t* __restrict__ cu,
                const uint8_t* __restrict__ has_init, int n_seq, int64_t n_tok, int n_heads,
                int n_qk, int n_slots, float eps, uint32_t* dev_err, int64_t n_items, int n_hgroups,
                const __grid_constant__ CUtensorMap xmap) {
  constexpr int NS = conv_stages<A>();
  constexpr int HALF = conv_half_bytes<A>();
  constexpr int TILE = conv_tile_bytes<A>();
  extern __shared__ __align__(128) uint8_t tiles[];      // NS x [CONV_ROWS][4 heads x 128] act
  __shared__ uint64_t bar[NS];                           // stage filled (copies complete)
  __shared__ uint64_t empty[NS];                         // stage read by all 16 warps
  __shared__ ConvItem meta[NS];
  __shared__ int abort_flag;
  __shared__ int64_t n_produced;                         // items of this block whose copies started
  constexpr int asz = A == BF16 ? 2 : 4;
  constexpr int ROW = CONV_HALF_COLS;                    // tile row stride in elements
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int C = n_heads * D;

  constexpr int WARPS = CONV_THREADS / 32;
  if (tid == 0) {
#pragma unroll
    for (int st = 0; st < NS; ++st) {
      tc::mbar_init(&bar[st], 1);
      tc::mbar_init(&empty[st], WARPS);
    }
    abort_flag = 0;
    n_produced = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();                                       // the barriers are initialised before any use

  // Warp 0: look up item `it` and start the copies of its tile into stage st.
  // Every call arrives once on the stage's barrier (with the byte count of the
  // copies, 0 for an item that stages nothing).
  auto produce = [&](int64_t it, int st) {
    ConvItem m{-1, 0, 0, 0, 0, 0, 0, 0, 0};
    const int j = (int)(it / n_hgroups), g = (int)(it % n_hgroups);
    int s = 0, ci = 0;
    int64_t t_chunk = 0;
    int n_here = 0, halves = 0;
    if (find_chunk(cu, n_seq, j, CHUNK, s, ci)) {
      m.s = s;
      m.ci = ci;
      m.head0 = g * CONV_HEADS_PER_BLOCK;
      const int slot = slot_idx[s];
      const int64_t seq0 = cu[s], seq1 = cu[s + 1];
      if (slot >= 0) {
        if (seq1 < seq0 || seq0 < 0 || seq1 > n_tok) m.flags = CI_BAD_SEQ;
        else if (slot >= n_slots) m.flags = CI_BAD_SLOT;
        else {
          m.flags = CI_VALID;
          t_chunk = seq0 + (int64_t)ci * CHUNK;
          n_here = (int)(min(t_chunk + CHUNK, seq1) - t_chunk);   // 0 only for an empty sequence
          m.slot = slot;
          m.n_here = n_here;
          m.t_chunk = t_chunk;
          m.seq0 = seq0;
          m.len = seq1 - seq0;
          if (ci > 0) m.flags |= CI_HALO_X;
          else if (has_init[s]) m.flags |= CI_HALO_STATE;
          halves = min(CONV_HEADS_PER_BLOCK, n_heads - m.head0) > 2 ? 2 : 1;
        }
      }
    }
    const bool halo = (m.flags & (CI_HALO_X | CI_HALO_STATE)) != 0;
    uint8_t* tile = tiles + (size_t)st * TILE;
    // one box of 64 rows per half (the whole box is counted, rows past the
    // chunk included), and 3 halo rows per half
    const int heads_here = m.flags & CI_VALID ? min(CONV_HEADS_PER_BLOCK, n_heads - m.head0) : 0;
    const uint32_t bytes = n_here > 0 ? (uint32_t)halves * CHUNK * ROW * asz : 0u;
    const uint32_t halo_bytes = halo ? (uint32_t)(KS * heads_here * D * asz) : 0u;   // exact channels
    const uint32_t w_bytes = (uint32_t)(heads_here * D * KW * asz);   // the item's conv_w rows
    if (lane == 0) {
      meta[st] = m;
      ++n_produced;
      tc::fence_async_smem();                            // earlier reads of the stage come first
      tc::mbar_arrive_expect_tx(&bar[st], bytes + halo_bytes + w_bytes);
      if (w_bytes)
        tc::bulk_load(tile + 2 * HALF, static_cast<const char*>(conv_w) + (size_t)m.head0 * D * KW * asz, w_bytes,
                      &bar[st]);
      for (int hf = 0; hf < halves && n_here > 0; ++hf)
        tma_box(tile + (size_t)hf * HALF + (size_t)KS * ROW * asz, &xmap, (m.head0 + 2 * hf) * D,
                (int)t_chunk, &bar[st]);
    }
    __syncwarp();                                        // the byte count is announced first
    if (halo && lane < 2 * KS && (lane & 1) < halves) {
      const int r = lane >> 1, hf = lane & 1;            // halo row r (0..2) of half hf
      const char* src;
      if (m.flags & CI_HALO_X)
        src = static_cast<const char*>(x) + ((t_chunk - KS + r) * ld_x + (int64_t)(m.head0 + 2 * hf) * D) * asz;
      else
        src = static_cast<const char*>(conv_state) +
              ((int64_t)slot_idx[s] * KS * C + (int64_t)r * C + (int64_t)(m.head0 + 2 * hf) * D) * asz;
      const uint32_t nb = (uint32_t)(min(2, heads_here - 2 * hf) * D * asz);   // the half's heads only
      tc::bulk_load(tile + (size_t)hf * HALF + (size_t)r * ROW * asz, src, nb, &bar[st]);
    }
    __syncwarp();
  };

  // Pipeline: item i of this block (it = blockIdx.x + i * gridDim.x) uses stage
  // i % NS; its copies complete phase i / NS of bar[stage], and phase i / NS of
  // empty[stage] completes when each of the 16 warps has finished reading it.
  // Warp 0 issues item i + NS - 1 at the start of item i, once item i - 1 (the
  // last user of that stage) has been released by every warp. No block-wide
  // barrier: the warps drift apart by up to the pipeline depth.
  const int64_t stride = gridDim.x;
  const int64_t n_mine_items = blockIdx.x < n_items ? (n_items - 1 - blockIdx.x) / stride + 1 : 0;
  if (warp == 0) {
    for (int64_t i = 0; i < NS - 1 && i < n_mine_items; ++i) produce(blockIdx.x + i * stride, (int)i);
  }

  const int grp = warp >> 1;
  const int hb = (warp & 1) * 2 + (lane >> 4);            // head within the item
  const int u0 = grp * CONV_TOK;                          // this thread's first token in the chunk
  bool failed = false;
  for (int64_t k = 0; k < n_mine_items; ++k) {
    if (warp == 0) {                                      // the item NS - 1 ahead goes in flight
      const int64_t i = k + NS - 1;
      if (i < n_mine_items) {
        const int sti = (int)(i % NS);
        bool ok = true;
        if (i >= NS) ok = tc::mbar_wait(&empty[sti], (uint32_t)((i / NS - 1) & 1), 1u << 24);
        if (__all_sync(FULL, ok)) produce(blockIdx.x + i * stride, sti);
        else failed = true;
      }
    }
    const int st = (int)(k % NS);
    if (!failed) failed = !tc::mbar_wait(&bar[st], (uint32_t)((k / NS) & 1), 1u << 24);
    if (failed || *reinterpret_cast<volatile int*>(&abort_flag)) {   // a wait gave up: stop
      if (lane == 0) {
        abort_flag = 1;
        report(dev_err, GDN_DEVERR_TIMEOUT);
      }
      break;
    }
    const ConvItem m = meta[st];
    if (!(m.flags & CI_VALID)) {
      if (m.ci == 0 && m.head0 == 0 && tid == 0 && m.flags)
        report(dev_err, m.flags & CI_BAD_SLOT ? GDN_DEVERR_SLOT : GDN_DEVERR_SEQLENS);
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[st]);          // this warp is done with the stage
      continue;
    }
    const uint8_t* tile = tiles + (size_t)st * TILE + (size_t)(warp & 1) * HALF;   // this warp's half
    const uint8_t* wtile = tiles + (size_t)st * TILE + 2 * HALF;                    // the item's conv_w rows
    const int slot = m.slot;
    const int64_t seq0 = m.seq0, len = m.len, t_chunk = m.t_chunk;
    const int n_here = m.n_here;
    const int heads_here = min(CONV_HEADS_PER_BLOCK, n_heads - m.head0);
    const int head = m.head0 + hb;
    const bool active = hb < heads_here;                  // uniform per 16 lanes
    const bool is_qk = head < 2 * n_qk;
    const int c0 = head * D + (lane & 15) * 8;            // global channel
    const int cb = (hb & 1) * D + (lane & 15) * 8;        // channel within a row of the half
    const int n_mine = max(0, min(CONV_TOK, n_here - u0)); // uniform per warp
    const bool zero_halo = u0 == 0 && !(m.flags & (CI_HALO_X | CI_HALO_STATE));

    if (n_mine > 0) {
      float2 w[4][4];                                     // [channel pair][tap]
      float2 p0[4], p1[4], p2[4];                         // the three previous rows
      {
        Raw8<A> wr[4];
        if (active) {
#pragma unroll
          for (int q = 0; q < 4; ++q) raw_load<A>(wtile, (int64_t)(c0 - m.head0 * D) * KW + 8 * q, wr[q]);
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) raw_zero<A>(wr[q]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {                     // channels 2q, 2q+1: 8 taps
          float t8[8];
          raw_unpack<A>(wr[q], t8);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) w[q][jj] = make_float2(t8[jj], t8[4 + jj]);
        }
        float r0[8], r1[8], r2[8];
        if (zero_halo) {                                  // chunk 0 without initial rows
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) { r0[jj] = 0.f; r1[jj] = 0.f; r2[jj] = 0.f; }
        } else {
          load8<A>(tile, (int64_t)u0 * ROW + cb, r0);    // tile rows u0 .. u0 + 2 = tokens u0 - 3 ..
          load8<A>(tile, (int64_t)(u0 + 1) * ROW + cb, r1);
          load8<A>(tile, (int64_t)(u0 + 2) * ROW + cb, r2);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          p0[q] = make_float2(r0[2 * q], r0[2 * q + 1]);
          p1[q] = make_float2(r1[2 * q], r1[2 * q + 1]);
          p2[q] = make_float2(r2[2 * q], r2[2 * q + 1]);
        }
      }
      // Conv + SiLU of all 8 tokens first (independent chains for the scheduler),
      // then the q/k norms of the 8 tokens together, then the stores. Tokens
      // past the chunk's end read stale tile rows; their values are discarded.
      float v[CONV_TOK][8], g[CONV_TOK];
#pragma unroll
      for (int u = 0; u < CONV_TOK; ++u) {
        float xv[8];
        load8<A>(tile, (int64_t)(u0 + u + KS) * ROW + cb, xv);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 cv = make_float2(xv[2 * q], xv[2 * q + 1]);
          const float2 a = silu2(conv4x2<A>(w[q][0], w[q][1], w[q][2], w[q][3], p0[q], p1[q], p2[q], cv));
          v[u][2 * q] = a.x;
          v[u][2 * q + 1] = a.y;
          p0[q] = p1[q]; p1[q] = p2[q]; p2[q] = cv;
        }
        if constexpr (NORM) g[u] = lane_sum_sq8(v[u]);
      }
      // The tile is read: release the stage now, so that its next copies start
      // while this warp takes the norms and stores (the loads, not the
      // arithmetic, set the item period).
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[st]);
      if constexpr (NORM) {
        if (__any_sync(FULL, is_qk)) {                  // warps of v heads only skip it
          const float r = lanes_inv_norm8(g, eps);      // tokens past n_mine: discarded
#pragma unroll
          for (int u = 0; u < CONV_TOK; ++u) {
            const float rn = __shfl_sync(FULL, r, (lane & 16) | token_lane(u));
            if (is_qk) {
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float2 o = __fmul2_rn(make_float2(v[u][2 * q], v[u][2 * q + 1]), make_float2(rn, rn));
                v[u][2 * q] = o.x;
                v[u][2 * q + 1] = o.y;
              }
            }
          }
        }
      }
      if (active) {
#pragma unroll
        for (int u = 0; u < CONV_TOK; ++u)
          if (u < n_mine) store8<A>(y, (t_chunk + u0 + u) * ld_y + c0, v[u]);
      }
    } else {
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[st]);          // nothing of the tile to read
    }

    // Final conv_state: rows len, len+1, len+2 of (initial rows ++ x rows),
    // written by the thread that read the initial rows (through the tile), after
    // its last read. When len < 3 new row r is old row len + r >= r; rows are
    // rewritten in ascending order, so each old row is read before it is
    // overwritten.
    if (m.ci == 0 && grp == 0 && active) {
      const bool hi = (m.flags & CI_HALO_STATE) != 0;
      const int64_t st_base = (int64_t)slot * KS * C;
#pragma unroll
      for (int r = 0; r < 3; ++r) {
        const int64_t idx = len + r;
        float v[8];
        if (idx >= 3) load8<A>(x, (seq0 + idx - 3) * ld_x + c0, v);
        else if (hi) load8<A>(conv_state, st_base + idx * C + c0, v);
        else {
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) v[jj] = 0.f;
        }
        store8<A>(conv_state, st_base + (int64_t)r * C + c0, v);
      }
    }
  }
  // Before the block exits no copy into its shared memory may still be in
  // flight: after a failed wait, wait (bounded) for the last copy of each stage.
  __syncthreads();
  if (abort_flag && warp == 0) {
    for (int64_t i = n_produced > NS ? n_produced - NS : 0; i < n_produced; ++i)
      tc::mbar_wait(&bar[i % NS], (uint32_t)((i / NS) & 1), 1u << 24);
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
static cudaError_t launch_conv_variant(unsigned grid, cudaStream_t stream, Args... args) {
  const int smem = conv_stages<A>() * conv_tile_bytes<A>();
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
  const int n_hgroups = (n_heads + CONV_HEADS_PER_BLOCK - 1) / CONV_HEADS_PER_BLOCK;
  // chunks of all sequences: at most ceil(n_tok / 64) + n_seq (every sequence,
  // empty ones too, owns at least one); items past the last chunk are skipped
  const int64_t max_chunks = (n_tok + CHUNK - 1) / CHUNK + n_seq;
  const int64_t n_items = max_chunks * n_hgroups;
  int n_sm = 0;
  cudaError_t e = sm_count(&n_sm);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(n_items < n_sm ? n_items : n_sm);   // one block per SM
  // x as a 2-D tensor [n_tok rows][C columns], row pitch ld_x, boxes of 256 x 64
  CUtensorMap xmap;
  {
    const EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const int es = cfg.act == GDN_BF16 ? 2 : 4;
    const cuuint64_t dims[2] = {(cuuint64_t)(n_heads * D), (cuuint64_t)(n_tok > 0 ? n_tok : 1)};
    const cuuint64_t strides[1] = {(cuuint64_t)ld_x * es};
    const cuuint32_t box[2] = {(cuuint32_t)CONV_HALF_COLS, (cuuint32_t)CHUNK};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(&xmap, cfg.act == GDN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                           2, const_cast<void*>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
#define GDN_CONV_ARGS                                                                     \
  x, ld_x, y, ld_y, conv_w, conv_state, slot_idx, cu, has_init, n_seq, n_tok, n_heads,   \
      cfg.n_qk_heads, cfg.n_slots, cfg.eps, cfg.dev_err, n_items, n_hgroups, xmap
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
