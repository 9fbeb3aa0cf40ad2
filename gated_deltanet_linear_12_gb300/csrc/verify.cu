// Read-only speculative verify of T = 1..8 draft tokens: conv of the draft rows
// from conv_state, SiLU, q/k L2 norm, the gated delta rule's output for every
// draft token from the current state, and the z-gated RMSNorm. The state and
// conv_state are only read (the accepted prefix is committed later by the
// batched commit, or at once by the decode mode of the step kernel).
//
// Source: "Strata PR #3226" ("Summary": the verify forward is launched once per
// GDN layer over all draft tokens) and the gated delta rule
// S_t = a_t S_{t-1}(I - b_t k_t k_t^T) + b_t v_t k_t^T, o_t = S_t q_t. The
// outputs come from the S0-product form (see step.cu): with the 2T products
// S0 k_t, S0 q_t of every value row, the deltas solve a unit lower-triangular
// system and o_t = g_t S0 q_t + sum_{s<=t} r(t,s) (k_s.q_t) d_s.
//
// Design (GB300). The step is a stream of 64 KiB f32 states, one per
// (sequence, v head), each read once; everything else is small. Two kernels:
//   verify_prep_kernel (one block of 128 threads per sequence and q/k head
//     group; all blocks fit on the GPU at once) does the state-independent
//     part: conv + SiLU + L2 norm of the group's q, k and v heads, the k.k and
//     q.k dot products and the gate tables of each v head. It writes the
//     post-conv rows, the tables and, for bf16 activations, the
//     [k_0..k_7 ; q_0..q_7] operand tile of the tensor-core product, all to a
//     caller-provided workspace.
//   verify_state_kernel (one block of 128 threads per sequence and v head;
//     thread r owns value row r) starts the four TMA copies of its state (boxes
//     of 32 columns x 128 rows, 128-byte swizzle) first, then waits for the prep
//     grid (programmatic dependent launch: the copies overlap the prep kernel)
//     and bulk-copies its small inputs behind them, all counted on one
//     mbarrier. Its critical path is one memory latency plus the arithmetic,
//     and three blocks fit on an SM. In the swizzled boxes row r of each box is
//     one 128-byte line whose 16-byte chunk c sits at c ^ (r mod 8), which
//     serves both arithmetic paths without a bank conflict:
//       - T = 1 (and f32 activations): thread r reads its row's chunks for the
//         dot products on the CUDA cores;
//       - T >= 2 with bf16 activations: thread r rewrites its own four lines in
//         place as bf16 hi | lo parts in the 128-byte-swizzled K-major operand
//         layout, and one tcgen05 product S0 [k_0..k_7 ; q_0..q_7]^T (M = 128,
//         N = 16, K = 128, two passes) gives all 2T dot products in TMEM.
// The dot products, the triangular solve and the epilogue are evaluated in the
// same order as the step kernel's, so at T = 1 the outputs are bitwise equal to
// those of the decode mode.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace gdn {

// The driver's tensor-map encoder, looked up once through the runtime.
EncodeTiledFn tensor_map_encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

cudaError_t encode_bf16_rows_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                                 uint64_t pitch, uint32_t box_cols, uint32_t box_rows) {
  const EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)(rows > 0 ? rows : 1)};
  const cuuint64_t strides[1] = {(cuuint64_t)pitch * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

VerifyWs verify_ws_layout(int B, int T, int Hk, int Hv, int act) {
  auto up = [](int64_t n) { return (n + 255) & ~(int64_t)255; };
  const int64_t C = (int64_t)(2 * Hk + Hv) * D;
  const int64_t asz = act == GDN_BF16 ? 2 : 4;
  VerifyWs w;
  w.act = 0;
  w.bt = up((int64_t)B * T * C * asz);
  w.tab = w.bt + up((int64_t)B * Hk * VERIFY_BT_BYTES);
  w.total = w.tab + up((int64_t)B * Hv * VERIFY_TAB_FLOATS * 4);
  return w;
}

namespace {

constexpr int VT = 128;                          // state kernel: thread r owns value row r
constexpr int PT = 128;                          // prep kernel threads
constexpr int S_BYTES = D * D * 4;               // one f32 state
constexpr int BT_BYTES = VERIFY_BT_BYTES;        // [k_0..7 ; q_0..7] bf16, K-major
constexpr int TAB = VERIFY_TAB_FLOATS;           // per (sequence, v head):
constexpr int TAB_A = 0;                         //   [8][8] b_t r(t,s) (k_t.k_s), s < t
constexpr int TAB_OC = 64;                       //   [8][8] r(t,s) (q_t.k_s), s <= t
constexpr int TAB_G = 128;                       //   [8] g_t
constexpr int TAB_BG = 136;                      //   [8] b_t g_t
constexpr int TAB_B = 144;                       //   [8] b_t
constexpr int QK_STRIDE = D + 4;                 // prep: padded f32 rows of q and k
constexpr int MAX_GROUP = 16;                    // v heads per q/k head (checked by the API)

// Byte offset of 16-byte chunk c (0..7) of line `line` (0..3) of row r: the
// state's box `line` holds columns 32 line .. 32 line + 31 (chunk c = columns
// 32 line + 4c ..), 16 KiB per box, 128 bytes per row, chunks swizzled by r mod 8.
// After the in-place conversion line 0 / 1 of row r holds its bf16 hi parts of
// columns 0..63 / 64..127 and line 2 / 3 the lo parts (chunk c = 8 columns).
__device__ __forceinline__ uint32_t line_off(int line, int r, int c) {
  return (uint32_t)(line * 16384 + r * 128 + ((c ^ (r & 7)) << 4));
}

// One TMA copy of a box of the state pool's 2-D view (128 columns x rows) into
// shared memory; completion is counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          tc::smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(tc::smem_u32(bar))
      : "memory");
}
// Programmatic dependent launch: let the next grid start / wait for the previous one.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Shared-memory descriptor of a bf16 K-major operand in the 128-byte swizzle
// layout (8-row groups 1024 bytes apart; the start address steps 32 bytes per
// K = 16 slice inside a 64-column atom).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  return tc::smem_desc(addr, 16, 1024) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ float4 unpack4(uint2 u) {
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

// ============================================================ prep kernel
// The dot product of two 128-vectors (padded f32 rows in shared memory) with the
// rounding of a warp dot product (lane l: x[4l] y[4l], then three fused
// multiply-adds; then an xor butterfly 16, 8, 4, 2, 1), evaluated by one thread.
__device__ __forceinline__ float dot128_as_warp(const float* a, const float* b) {
  float part[32];
#pragma unroll
  for (int l = 0; l < 32; ++l) {
    const float4 x = reinterpret_cast<const float4*>(a)[l];
    const float4 y = reinterpret_cast<const float4*>(b)[l];
    float p = __fmul_rn(x.x, y.x);
    p = __fmaf_rn(x.y, y.y, p);
    p = __fmaf_rn(x.z, y.z, p);
    p = __fmaf_rn(x.w, y.w, p);
    part[l] = p;
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1)
#pragma unroll
    for (int l = 0; l < m; ++l) part[l] = __fadd_rn(part[l], part[l + m]);
  return part[0];
}

template <int A>
__global__ void __launch_bounds__(PT, 4) verify_prep_kernel(StepArgs p, uint8_t* __restrict__ ws, VerifyWs wl,
                                                            void* __restrict__ act_rows) {
  pdl_launch_dependents();                               // the state kernel may start its copies
  __shared__ __align__(16) float q_s[MAXT * QK_STRIDE];
  __shared__ __align__(16) float k_s[MAXT * QK_STRIDE];
  __shared__ float kk_s[MAXT * MAXT], qk_s[MAXT * MAXT];
  __shared__ float al_s[MAX_GROUP * MAXT], be_s[MAX_GROUP * MAXT];
  const int tid = threadIdx.x;
  const int hq = blockIdx.x, b = blockIdx.y;
  const int T = p.T, Hk = p.Hk, Hv = p.Hv, G = Hv / Hk, h0 = hq * G, nh = 2 + G;
  const int C = (2 * Hk + Hv) * D;
  const int slot = p.slot_idx[b];
  if (slot < 0) return;                                   // padding entry
  if (slot >= p.n_slots) {
    if (tid == 0 && hq == 0) report(p.dev_err, GDN_DEVERR_SLOT);
    return;
  }

  // ---- post-conv activations. Item (part, head, l16): 8 channels of head `head`
  // (0 q, 1 k, 2.. v) for tokens 4 part .. 4 part + 3; rows t..t+3 of
  // (conv_state rows ++ draft rows) feed token t. 16-lane groups share (part, head).
  // The gates are loaded behind the rows and staged after the conv.
  {
    const int n_parts = (T + 3) / 4;
    const int n_items = n_parts * nh * 16;
    const int64_t xb = (int64_t)b * T * C;
    const int64_t cs = (int64_t)slot * KS * C;
    for (int base = 0; base < n_items; base += PT) {      // uniform trip count
      const int item = base + tid;
      const bool grp = item < n_items;                    // uniform per 16 lanes
      const int l16 = item & 15, head = (item >> 4) % nh, part = (item >> 4) / nh;
      const int t0 = 4 * part;
      const int c = (head == 0 ? hq * D : head == 1 ? (Hk + hq) * D : (2 * Hk + h0 + head - 2) * D) + l16 * 8;
      Raw8<A> wr[4], rw[7];
      if (grp) {
#pragma unroll
        for (int q = 0; q < 4; ++q) raw_load<A>(p.conv_w, (int64_t)c * KW + 8 * q, wr[q]);
#pragma unroll
        for (int j = 0; j < 7; ++j) {
          const int idx = t0 + j;
          if (idx < KS) raw_load<A>(p.conv_state, cs + (int64_t)idx * C + c, rw[j]);
          else if (idx - KS < T) raw_load<A>(p.x, xb + (int64_t)(idx - KS) * C + c, rw[j]);
          else raw_zero<A>(rw[j]);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) raw_zero<A>(wr[q]);
#pragma unroll
        for (int j = 0; j < 7; ++j) raw_zero<A>(rw[j]);
      }
      float ga = 0.f, gb = 0.f;                           // this thread's gate pair, if any
      const bool gate = base == 0 && tid < G * T;         // G * T <= 128 = PT
      if (gate) {
        const int64_t gi = ((int64_t)b * T + tid % T) * Hv + h0 + tid / T;
        ga = p.alpha[gi];
        gb = p.beta[gi];
      }
      float2 w[4][4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float t8[8];
        raw_unpack<A>(wr[q], t8);
#pragma unroll
        for (int j = 0; j < 4; ++j) w[q][j] = make_float2(t8[j], t8[4 + j]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int t = t0 + u;
        const bool live = grp && t < T;
        float v[8];
        if (live) {
          float r0[8], r1[8], r2[8], r3[8];
          raw_unpack<A>(rw[u], r0);
          raw_unpack<A>(rw[u + 1], r1);
          raw_unpack<A>(rw[u + 2], r2);
          raw_unpack<A>(rw[u + 3], r3);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 a = silu2(conv4x2(w[q][0], w[q][1], w[q][2], w[q][3],
                                           make_float2(r0[2 * q], r0[2 * q + 1]),
                                           make_float2(r1[2 * q], r1[2 * q + 1]),
                                           make_float2(r2[2 * q], r2[2 * q + 1]),
                                           make_float2(r3[2 * q], r3[2 * q + 1])));
            v[2 * q] = a.x;
            v[2 * q + 1] = a.y;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = 0.f;
        }
        const float ss = head_sum_sq16(v);                // all 32 lanes of the warp
        if (live && head < 2) {
          const float r = inv_norm(ss, p.eps);
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = __fmul_rn(v[j], r);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = round_act<A>(v[j]);
        if (live) {
          store8<A>(act_rows, xb + (int64_t)t * C + c, v);
          if (head < 2) {
            float* dst = (head == 0 ? q_s : k_s) + t * QK_STRIDE + l16 * 8;
            reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
            reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
          }
        }
      }
      if (gate) {
        al_s[(tid / T) * MAXT + tid % T] = ga;
        be_s[(tid / T) * MAXT + tid % T] = gb;
      }
    }
  }
  __syncthreads();

  // ---- k.k and q.k dot products (one pair per thread), the operand tile
  {
    const int which = tid >> 6, t = (tid >> 3) & 7, s = tid & 7;   // 0: k.k (s < t), 1: q.k (s <= t)
    if (t < T && (which == 0 ? s < t : s <= t)) {
      const float d = dot128_as_warp((which == 0 ? k_s : q_s) + t * QK_STRIDE, k_s + s * QK_STRIDE);
      (which == 0 ? kk_s : qk_s)[t * MAXT + s] = d;
    }
  }
  if constexpr (A == BF16) {                              // 16 rows x 16 chunks of 8, K-major
    for (int e = tid; e < 256; e += PT) {
      const int row = e >> 4, kc = e & 15, t = row & 7;
      uint32_t wd[4] = {0u, 0u, 0u, 0u};
      if (t < T) {
        const float* src = (row < 8 ? k_s : q_s) + t * QK_STRIDE + 8 * kc;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(src[2 * j], src[2 * j + 1]);
          wd[j] = *reinterpret_cast<const uint32_t*>(&h2);
        }
      }
      uint8_t* bt = ws + wl.bt + ((int64_t)b * Hk + hq) * BT_BYTES;
      *reinterpret_cast<uint4*>(bt + tc::kmajor_offset(row, 8 * kc, 16)) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
    }
  }
  __syncthreads();

  // ---- gate tables of each v head of the group; products in ascending order
  // (r(t,s) = a_{s+1} ... a_t, g_t = a_0 ... a_t)
  for (int e = tid; e < G * MAXT * MAXT; e += PT) {
    const int g = e >> 6, t = (e >> 3) & 7, s = e & 7;
    if (t >= T || s > t) continue;
    const float* al = al_s + g * MAXT;
    float* tab = reinterpret_cast<float*>(ws + wl.tab) + ((int64_t)b * Hv + h0 + g) * TAB;
    float r = 1.f;
    for (int u = s + 1; u <= t; ++u) r = __fmul_rn(r, al[u]);
    const float bt = be_s[g * MAXT + t];
    if (s < t) tab[TAB_A + t * MAXT + s] = __fmul_rn(__fmul_rn(bt, r), kk_s[t * MAXT + s]);
    tab[TAB_OC + t * MAXT + s] = __fmul_rn(r, qk_s[t * MAXT + s]);
    if (s == 0) {
      float gt = al[0];
      for (int u = 1; u <= t; ++u) gt = __fmul_rn(gt, al[u]);
      tab[TAB_G + t] = gt;
      tab[TAB_BG + t] = __fmul_rn(bt, gt);
      tab[TAB_B + t] = bt;
    }
  }
}

// ============================================================ state kernel
// Shared memory: the state (then its hi | lo parts, then the outputs), the
// operand tile (bf16) or k and q rows (f32), v rows, z rows, the table row, norm_w.
template <int A> __host__ __device__ constexpr int qk_bytes() { return A == BF16 ? BT_BYTES : 2 * MAXT * D * 4; }
template <int A> __host__ __device__ constexpr int rows_bytes() { return MAXT * D * (A == BF16 ? 2 : 4); }
template <int A> __host__ __device__ constexpr int state_smem() {
  return S_BYTES + qk_bytes<A>() + 2 * rows_bytes<A>() + TAB * 4 + D * 4;
}

// Activations k_t (which = 0) or q_t (which = 1), columns 4j..4j+3: bf16 from
// the operand tile (k_t row t, q_t row 8 + t), f32 from the k | q rows.
template <int A>
__device__ __forceinline__ float4 act4(const uint8_t* QK, int which, int t, int j) {
  if constexpr (A == BF16) {
    return unpack4(*reinterpret_cast<const uint2*>(QK + tc::kmajor_offset(8 * which + t, 4 * j, 16)));
  } else {
    return reinterpret_cast<const float4*>(QK + which * MAXT * D * 4)[t * (D / 4) + j];
  }
}
template <int A> __device__ __forceinline__ float row_at(const uint8_t* R, int t, int i) {
  if constexpr (A == BF16) return bf2f(reinterpret_cast<const uint16_t*>(R)[t * D + i]);
  else return reinterpret_cast<const float*>(R)[t * D + i];
}

// NT > 0: the number of draft tokens as a compile-time constant (CUDA-core
// variants; keeps the unrolled code small enough for the instruction cache);
// NT = 0: read from the arguments.
template <int A, bool TC, int NT>
__global__ void __launch_bounds__(VT, 3)
verify_state_kernel(StepArgs p, const __grid_constant__ CUtensorMap smap, const uint8_t* __restrict__ ws,
                    VerifyWs wl, const void* __restrict__ act_rows) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x, b = blockIdx.y;
  const int T = NT > 0 ? NT : p.T;
  const int Hk = p.Hk, Hv = p.Hv, G = Hv / Hk, hq = h / G;
  const int C = (2 * Hk + Hv) * D;
  const int slot = p.slot_idx[b];
  if (slot < 0 || slot >= p.n_slots) return;              // padding, or reported by the prep kernel

  uint8_t* SR = smem;                                     // state -> hi | lo -> outputs
  uint8_t* QK = SR + S_BYTES;                             // operand tile (bf16) / k, q rows (f32)
  uint8_t* VR = QK + qk_bytes<A>();                       // v rows [T][128]
  uint8_t* ZR = VR + rows_bytes<A>();                     // z rows [T][128]
  float* tb = reinterpret_cast<float*>(ZR + rows_bytes<A>());       // the table row
  float* nw = tb + TAB;                                              // norm_w
  constexpr int asz = A == BF16 ? 2 : 4;
  constexpr uint32_t row_bytes = D * asz;

  __shared__ uint64_t s_bar, tc_bar;
  __shared__ uint32_t tc_slot;
  if (tid == 0) {
    tc::mbar_init(&s_bar, 1);
    if constexpr (TC) tc::mbar_init(&tc_bar, 1);
    tc::fence_mbar_init();
    tc::fence_async_smem();
  }
  if constexpr (TC) {
    if (warp == 1) {
      tc::tmem_alloc(&tc_slot, 32);
      tc::tmem_relinquish();
    }
  }
  __syncthreads();                                        // barriers initialised before any wait
  // ---- the state first (independent of the prep kernel), then the rest
  if (warp == 0) {
    if (lane == 0) {
      const uint32_t bytes =
          S_BYTES + (A == BF16 ? BT_BYTES : 2u * T * row_bytes) + 2u * T * row_bytes + TAB * 4 + D * 4;
      tc::mbar_arrive_expect_tx(&s_bar, bytes);
      const int row0 = (slot * Hv + h) * D;
#pragma unroll
      for (int bx = 0; bx < 4; ++bx) tma_load_2d(SR + bx * 16384, &smap, 32 * bx, row0, &s_bar);
    }
    __syncwarp();
    pdl_wait();                                           // the prep kernel's rows and tables
    const char* act = static_cast<const char*>(act_rows);
    const char* zp = static_cast<const char*>(p.z);
    if (lane < T) {
      const int t = lane;
      const int64_t tok = (int64_t)b * T + t;
      tc::bulk_load(VR + t * row_bytes, act + (tok * C + (int64_t)(2 * Hk + h) * D) * asz, row_bytes, &s_bar);
      tc::bulk_load(ZR + t * row_bytes, zp + (tok * Hv * D + (int64_t)h * D) * asz, row_bytes, &s_bar);
      if constexpr (A != BF16) {
        tc::bulk_load(QK + t * row_bytes, act + (tok * C + (int64_t)(Hk + hq) * D) * asz, row_bytes, &s_bar);
        tc::bulk_load(QK + MAXT * row_bytes + t * row_bytes, act + (tok * C + (int64_t)hq * D) * asz, row_bytes,
                  &s_bar);
      }
    } else if (lane == 8) {
      tc::bulk_load(tb, ws + wl.tab + ((int64_t)b * Hv + h) * TAB * 4, TAB * 4, &s_bar);
    } else if (lane == 9) {
      if constexpr (A == BF16) tc::bulk_load(QK, ws + wl.bt + ((int64_t)b * Hk + hq) * BT_BYTES, BT_BYTES, &s_bar);
    } else if (lane == 10) {
      tc::bulk_load(nw, p.norm_w, D * 4, &s_bar);
    }
  }
  const bool s_ok = tc::mbar_wait(&s_bar, 0, 1u << 24);
  if constexpr (TC) tc::fence_before_sync();
  const bool s_failed = __syncthreads_or(!s_ok);
  bool failed = s_failed;

  const int r = tid;                                      // value row
  float sk[MAXT], sq[MAXT];
  uint32_t tbase = 0;
  if (failed) {
    // error exit below
  } else if constexpr (TC) {
    // row r as bf16 hi | lo in place: columns 0..63 (lines 0, 1) give hi -> line 0
    // and lo -> line 2; columns 64..127 (lines 2, 3) give hi -> line 1 and
    // lo -> line 3. Every line is read before it is overwritten.
    float x[64];
    uint4 hi[8], lo[8];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const float4 f = *reinterpret_cast<const float4*>(SR + line_off(c >> 3, r, c & 7));
      x[4 * c] = f.x; x[4 * c + 1] = f.y; x[4 * c + 2] = f.z; x[4 * c + 3] = f.w;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) tc::split8(x + 8 * c, hi[c], lo[c]);
#pragma unroll
    for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(SR + line_off(0, r, c)) = hi[c];
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const float4 f = *reinterpret_cast<const float4*>(SR + line_off(2 + (c >> 3), r, c & 7));
      x[4 * c] = f.x; x[4 * c + 1] = f.y; x[4 * c + 2] = f.z; x[4 * c + 3] = f.w;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(SR + line_off(2, r, c)) = lo[c];
#pragma unroll
    for (int c = 0; c < 8; ++c) tc::split8(x + 8 * c, hi[c], lo[c]);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      *reinterpret_cast<uint4*>(SR + line_off(1, r, c)) = hi[c];
      *reinterpret_cast<uint4*>(SR + line_off(3, r, c)) = lo[c];
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    tbase = tc_slot;
    if (tid == 0) {
      const uint32_t sh = tc::smem_u32(SR), sl = sh + 32768, bt = tc::smem_u32(QK);
      const uint32_t id = tc::idesc_bf16_f32(128, 16);
#pragma unroll 1
      for (int ks = 0; ks < 8; ++ks)
        tc::mma_bf16(tbase, smem_desc_sw128(sh + (ks >> 2) * 16384 + (ks & 3) * 32),
                     tc::smem_desc(bt + ks * 512, 256, 128), id, ks > 0);
#pragma unroll 1
      for (int ks = 0; ks < 8; ++ks)
        tc::mma_bf16(tbase, smem_desc_sw128(sl + (ks >> 2) * 16384 + (ks & 3) * 32),
                     tc::smem_desc(bt + ks * 512, 256, 128), id, 1);
      tc::mma_commit(&tc_bar);
    }
    const bool ok = tc::mbar_wait(&tc_bar, 0, 1u << 24);
    tc::fence_after_sync();
    failed = __syncthreads_or(!ok);
    if (!failed) {
      float acc[16];
      tc::tmem_ld16(tbase + ((uint32_t)(32 * warp) << 16), acc);
#pragma unroll
      for (int t = 0; t < MAXT; ++t) { sk[t] = acc[t]; sq[t] = acc[8 + t]; }
    }
  } else {
    // row r on the CUDA cores, with the step kernel's rounding: four partial sums
    // over the chunks j = 4m + cg (m ascending), then (p0 + p1) + (p2 + p3)
    float pk[MAXT][4], pq[MAXT][4];
#pragma unroll
    for (int t = 0; t < MAXT; ++t)
#pragma unroll
      for (int cg = 0; cg < 4; ++cg) { pk[t][cg] = 0.f; pq[t][cg] = 0.f; }
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int cg = j & 3;
      const float4 s4 = *reinterpret_cast<const float4*>(SR + line_off(j >> 3, r, j & 7));
#pragma unroll
      for (int t = 0; t < MAXT; ++t) {
        if (t < T) {
          const float4 k = act4<A>(QK, 0, t, j);
          float a = pk[t][cg];
          a = __fmaf_rn(s4.x, k.x, a); a = __fmaf_rn(s4.y, k.y, a);
          a = __fmaf_rn(s4.z, k.z, a); a = __fmaf_rn(s4.w, k.w, a);
          pk[t][cg] = a;
          const float4 q = act4<A>(QK, 1, t, j);
          float c = pq[t][cg];
          c = __fmaf_rn(s4.x, q.x, c); c = __fmaf_rn(s4.y, q.y, c);
          c = __fmaf_rn(s4.z, q.z, c); c = __fmaf_rn(s4.w, q.w, c);
          pq[t][cg] = c;
        }
      }
    }
#pragma unroll
    for (int t = 0; t < MAXT; ++t) {
      sk[t] = __fadd_rn(__fadd_rn(pk[t][0], pk[t][1]), __fadd_rn(pk[t][2], pk[t][3]));
      sq[t] = __fadd_rn(__fadd_rn(pq[t][0], pq[t][1]), __fadd_rn(pq[t][2], pq[t][3]));
    }
  }

  if (failed) {                    // a completion wait gave up: no outputs for this state
    if (tid == 0) report(p.dev_err, GDN_DEVERR_TIMEOUT);
    if (s_failed) tc::mbar_wait(&s_bar, 0, 1u << 24);   // the copies, if still in flight
    if constexpr (TC) {
      if (!s_failed) tc::mbar_wait(&tc_bar, 0, 1u << 24);   // the product in flight
      tc::fence_before_sync();
      __syncthreads();
      if (warp == 1) tc::tmem_dealloc(tc_slot, 32);
    }
    return;
  }

  // ---- deltas and outputs of row r (the step kernel's order)
  float o[MAXT];
  {
    float dr[MAXT];
#pragma unroll
    for (int t = 0; t < MAXT; ++t) {
      if (t < T) {
        float x = __fmaf_rn(-tb[TAB_BG + t], sk[t], __fmul_rn(tb[TAB_B + t], row_at<A>(VR, t, r)));
#pragma unroll
        for (int u = 0; u < t; ++u) x = __fmaf_rn(-tb[TAB_A + t * MAXT + u], dr[u], x);
        dr[t] = x;
        float y = __fmul_rn(tb[TAB_G + t], sq[t]);
#pragma unroll
        for (int u = 0; u <= t; ++u) y = __fmaf_rn(tb[TAB_OC + t * MAXT + u], dr[u], y);
        o[t] = __fmul_rn(y, p.q_scale);
      }
    }
  }
  if constexpr (TC) tc::fence_before_sync();
  __syncthreads();                                        // the state region is free
  float* o_s = reinterpret_cast<float*>(SR);
#pragma unroll
  for (int t = 0; t < MAXT; ++t)
    if (t < T) o_s[t * D + r] = o[t];
  __syncthreads();

  // ---- z-gated RMSNorm: one 16-lane group per token
  {
    const int t = tid >> 4, l16 = tid & 15;
    const bool live = t < T;
    float ov[8];
    if (live) {
      const float4 u0 = reinterpret_cast<const float4*>(o_s + t * D)[2 * l16];
      const float4 u1 = reinterpret_cast<const float4*>(o_s + t * D)[2 * l16 + 1];
      ov[0] = u0.x; ov[1] = u0.y; ov[2] = u0.z; ov[3] = u0.w;
      ov[4] = u1.x; ov[5] = u1.y; ov[6] = u1.z; ov[7] = u1.w;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) ov[j] = 0.f;
    }
    const float ss = head_sum_sq16(ov);
    if (live) {
      const float rn = inv_norm(__fmul_rn(ss, 1.0f / D), p.eps);
      float zv[8], res[8];
      load8<A>(ZR, (int64_t)t * D + l16 * 8, zv);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        res[j] = __fmul_rn(__fmul_rn(__fmul_rn(ov[j], rn), nw[l16 * 8 + j]), silu_gate(zv[j]));
      store8<A>(p.out, ((int64_t)b * T + t) * Hv * D + (int64_t)h * D + l16 * 8, res);
    }
  }
  if constexpr (TC) {
    if (warp == 1) tc::tmem_dealloc(tbase, 32);
  }
}

// ------------------------------------------------------------------ host side

// The state pool as a 2-D f32 tensor of 128 columns and n_slots * Hv * 128 rows,
// copied in boxes of 32 columns x 128 rows with the 128-byte swizzle.
cudaError_t state_map(const StepArgs& a, CUtensorMap* m) {
  const EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const uint64_t rows = (uint64_t)a.n_slots * (uint64_t)a.Hv * D;
  if (rows > 0x7fffffffull) return cudaErrorInvalidValue;        // TMA row coordinates are int32
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)D * sizeof(float)};
  const cuuint32_t box[2] = {32, (cuuint32_t)D};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.state, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int A, bool TC, int NT>
cudaError_t launch_state(const StepArgs& a, const CUtensorMap& smap, const uint8_t* ws, const VerifyWs& wl,
                         const void* act_rows, cudaStream_t stream) {
  auto kern = verify_state_kernel<A, TC, NT>;
  const int smem = state_smem<A>();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hv, a.B);
  cfg.blockDim = dim3(VT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, smap, ws, wl, act_rows);
}

template <int A>
cudaError_t launch_pair(const StepArgs& a, uint8_t* ws, cudaStream_t stream) {
  const VerifyWs wl = verify_ws_layout(a.B, a.T, a.Hk, a.Hv, A);
  void* act_rows = a.postconv ? a.postconv : static_cast<void*>(ws + wl.act);
  CUtensorMap smap;
  cudaError_t e = state_map(a, &smap);
  if (e != cudaSuccess) return e;
  verify_prep_kernel<A><<<dim3(a.Hk, a.B), PT, 0, stream>>>(a, ws, wl, act_rows);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if constexpr (A == BF16) {
    return a.T >= 2 ? launch_state<A, true, 0>(a, smap, ws, wl, act_rows, stream)
                    : launch_state<A, false, 1>(a, smap, ws, wl, act_rows, stream);
  } else {
    switch (a.T) {
      case 1: return launch_state<A, false, 1>(a, smap, ws, wl, act_rows, stream);
      case 2: return launch_state<A, false, 2>(a, smap, ws, wl, act_rows, stream);
      case 3: return launch_state<A, false, 3>(a, smap, ws, wl, act_rows, stream);
      case 4: return launch_state<A, false, 4>(a, smap, ws, wl, act_rows, stream);
      case 5: return launch_state<A, false, 5>(a, smap, ws, wl, act_rows, stream);
      case 6: return launch_state<A, false, 6>(a, smap, ws, wl, act_rows, stream);
      case 7: return launch_state<A, false, 7>(a, smap, ws, wl, act_rows, stream);
      default: return launch_state<A, false, 8>(a, smap, ws, wl, act_rows, stream);
    }
  }
}

}  // namespace

// bf16 activations with two or more draft tokens take the tensor-core product;
// T = 1 and f32 activations the CUDA-core rows.
cudaError_t launch_verify_readonly(const StepArgs& a, int act, void* ws, cudaStream_t stream) {
  return act == GDN_BF16 ? launch_pair<BF16>(a, static_cast<uint8_t*>(ws), stream)
                         : launch_pair<F32>(a, static_cast<uint8_t*>(ws), stream);
}

}  // namespace gdn
