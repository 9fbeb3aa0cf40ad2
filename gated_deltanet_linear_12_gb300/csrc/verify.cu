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
// (sequence, v head), each read once; everything else is small. One kernel per
// layer, one block of 128 threads per (sequence, v head), three blocks per SM
// (76.5 KB of shared memory each); thread r owns value row r. The state comes
// in four TMA boxes of 32 columns x 128 rows with the 128-byte swizzle: row r of
// a box is one 128-byte line whose 16-byte chunk c sits at c ^ (r mod 8), which
// is both a bank-conflict-free row for thread r and the canonical K-major
// operand layout of the tensor core. The block computes its q, k and v conv rows
// itself (the two v heads of a q/k head each redo the q, k part: sharing it
// through memory was measured slower); thread r convolves v channel r itself, so
// v_t[r] stays in its registers. The activations enter the recurrence unrounded
// (f32); only the optional post-conv copy is rounded to the activation dtype.
// Then
//   - T <= 4 (and f32 activations): the 2T dot products of every row on the CUDA
//     cores, in the step kernel's order, so that at T = 1 the outputs are
//     bitwise equal to those of the decode mode;
//   - T >= 5 with bf16 activations: one tcgen05 kind::tf32 product
//     S0 [k_0..k_7 ; q_0..q_7]^T straight from the boxes (the state and k, q are
//     read as tf32: 10 explicit mantissa bits); the k.k and q.k dot products on
//     the CUDA cores while the state is still arriving.
// Launched as a programmatic dependent launch: a block that becomes resident
// while the previous grid drains sets up before it waits; in the CUDA-core
// variants it also asks L2 for its state and for the rows of the block one wave
// later. The small loads of the conv go out before the state's 64 KiB copy:
// queued behind the copy they arrive late, and every phase waits on them.
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

namespace {

constexpr int VT = 128;                          // state kernel: thread r owns value row r
constexpr int S_BYTES = D * D * 4;               // one f32 state
constexpr int TAB = 160;                         // per (sequence, v head):
constexpr int TAB_A = 0;                         //   [8][8] b_t r(t,s) (k_t.k_s), s < t
constexpr int TAB_OC = 64;                       //   [8][8] r(t,s) (q_t.k_s), s <= t
constexpr int TAB_G = 128;                       //   [8] g_t
constexpr int TAB_BG = 136;                      //   [8] b_t g_t
constexpr int TAB_B = 144;                       //   [8] b_t

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

// Shared-memory descriptor of a bf16 K-major operand in the 128-byte swizzle
// layout (8-row groups 1024 bytes apart; the start address steps 32 bytes per
// K = 16 slice inside a 64-column atom).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
  return tc::smem_desc(addr, 16, 1024) | ((uint64_t)2 << 61);
}

// ============================================================ the verify kernel
// Shared memory (no static shared variables, so the dynamic region starts at a
// 1024-byte boundary):
//   QK  q and k of every draft token, f32 [k_0..k_7 ; q_0..q_7], K-major with the
//       128-byte swizzle (the tf32 operand of the tensor-core variant; float4
//       reads without conversion for the CUDA-core ones); after the products
//       the outputs o_t (f32 [T][128])
//   SR  the state, four TMA boxes [32 columns][128 rows] f32, 128-byte swizzle
//       (1024-byte aligned)
//   VS  v rows [T][128] f32 (CUDA-core variants; the tensor-core one keeps v in
//       registers)
//   TB  the table of gate products and dot products (TAB floats)
//   GS  alpha, beta of this head [2][8]
//   BR  the state and product barriers (and an unused one), the TMEM address, the
//       issued flag
template <int A, bool TC> __host__ __device__ constexpr int qk_bytes() { return 2 * MAXT * D * 4; }
template <int A, bool TC> __host__ __device__ constexpr int qk_region() { return (qk_bytes<A, TC>() + 1023) & ~1023; }
// Where the v rows live: shared memory [NT][128] f32 for the CUDA-core variants
// of up to 4 draft tokens; registers (thread r keeps v_t[r]) for the others,
// whose 8 rows of f32 would not fit three bf16 blocks per SM.
template <bool TC, int NT> __host__ __device__ constexpr bool v_in_regs() { return TC || NT == 0 || NT > 4; }
template <bool TC, int NT> __host__ __device__ constexpr int vs_bytes() { return v_in_regs<TC, NT>() ? 0 : NT * D * 4; }
template <int A, bool TC, int NT> __host__ __device__ constexpr int verify_smem() {
  return qk_region<A, TC>() + S_BYTES + vs_bytes<TC, NT>() + TAB * 4 + 2 * MAXT * 4 + 32;
}

// Byte offset of f32 element (row, k) of the [16][128] tf32 operand in the
// 128-byte-swizzled K-major layout: K blocks of 32 columns, 2048 bytes each (two
// 8-row groups of 1024 bytes), 128 bytes per row, 16-byte chunk c of row r at
// chunk c ^ (r mod 8).
__device__ __forceinline__ uint32_t bsw_off(int row, int k) {
  return (uint32_t)((k >> 5) * 2048 + (row >> 3) * 1024 + (row & 7) * 128 + ((((k & 31) >> 2) ^ (row & 7)) << 4) +
                    (k & 3) * 4);
}

// Activations k_t (which = 0) or q_t (which = 1), columns 4j..4j+3.
template <int A, bool TC>
__device__ __forceinline__ float4 act4(const uint8_t* QK, int which, int t, int j) {
  return *reinterpret_cast<const float4*>(QK + bsw_off(8 * which + t, 4 * j));
}

// Stores 8 rounded activations (columns c .. c + 7) of k_t (which = 0) or q_t.
template <int A, bool TC>
__device__ __forceinline__ void put_act8(uint8_t* QK, int which, int t, int c, const float v[8]) {
  *reinterpret_cast<float4*>(QK + bsw_off(8 * which + t, c)) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(QK + bsw_off(8 * which + t, c + 4)) = make_float4(v[4], v[5], v[6], v[7]);
}

// One activation of `base` as raw bits (bf16 in the low half, or the f32 bits),
// widened later: a load whose value is not used at once does not stall the loads
// after it; and one activation stored (rounded) from f32.
template <int A> __device__ __forceinline__ uint32_t load1_bits(const void* base, int64_t i) {
  if constexpr (A == BF16) return static_cast<const uint16_t*>(base)[i];
  else return static_cast<const uint32_t*>(base)[i];
}
template <int A> __device__ __forceinline__ float bits_to_f(uint32_t b) {
  if constexpr (A == BF16) return __uint_as_float(b << 16);
  else return __uint_as_float(b);
}
template <int A> __device__ __forceinline__ void store1(void* base, int64_t i, float v) {
  if constexpr (A == BF16) static_cast<uint16_t*>(base)[i] = f2bf(v);
  else static_cast<float*>(base)[i] = v;
}

// Programmatic dependent launch: let the next grid start / wait for the previous one.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// A hint: start bringing a box of the state pool into L2 (no completion, no fault
// on out-of-range boxes).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y)
               : "memory");
}

// The sum (a0 + a1) + (a2 + a3) of four TMEM accumulators of 16 columns each at
// taddr, taddr + 16, taddr + 32, taddr + 48 (this warp's 32 lanes).
__device__ __forceinline__ void sum4_ld16(uint32_t taddr, float v[16]) {
  float a[16], b2[16], c[16], d[16];
  tc::tmem_ld16x4(taddr, a, taddr + 16, b2, taddr + 32, c, taddr + 48, d);
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __fadd_rn(__fadd_rn(a[i], b2[i]), __fadd_rn(c[i], d[i]));
}

// L2 hints for unit u = b Hv + h (sequence b, v head h); the slot index read
// here may still change: nothing but these hints depends on it.
// hint_state: box `box` (0..3) of its state.
__device__ __forceinline__ void hint_state(const StepArgs& p, const CUtensorMap* smap, int u, int box) {
  const int Hv = p.Hv, b = u / Hv, h = u % Hv;
  const int slot = *reinterpret_cast<const volatile int32_t*>(p.slot_idx + b);
  if (slot >= 0 && slot < p.n_slots) tma_prefetch_2d(smap, 32 * box, (slot * Hv + h) * D);
}
// hint_rows: row w (0 <= w < 3 (T + 3) + T) of its conv rows (conv_state and x
// rows of its q, k and v heads), then its z rows.
template <int A>
__device__ __forceinline__ void hint_rows(const StepArgs& p, int u, int T, int w) {
  const int Hk = p.Hk, Hv = p.Hv, G = Hv / Hk, C = (2 * Hk + Hv) * D;
  const int b = u / Hv, h = u % Hv, hq = h / G;
  const int n_x = (T + KS) * 3;
  if (w < 0 || w >= n_x + T) return;
  const int slot = *reinterpret_cast<const volatile int32_t*>(p.slot_idx + b);
  if (slot < 0 || slot >= p.n_slots) return;
  constexpr int esz = A == BF16 ? 2 : 4;
  if (w < n_x) {
    const int row = w / 3, hd = w % 3;
    const int64_t c = hd == 0 ? (int64_t)hq * D : hd == 1 ? (int64_t)(Hk + hq) * D : (int64_t)(2 * Hk + h) * D;
    const int64_t e = row < KS ? ((int64_t)slot * KS + row) * C + c : ((int64_t)b * T + row - KS) * C + c;
    tc::prefetch_l2((row < KS ? static_cast<const char*>(p.conv_state) : static_cast<const char*>(p.x)) + e * esz,
                D * esz);
  } else {
    const int t = w - n_x;
    tc::prefetch_l2(static_cast<const char*>(p.z) + (((int64_t)b * T + t) * Hv + h) * D * esz, D * esz);
  }
}

// Resident blocks per SM (shared memory at most 74.7 KiB per bf16 block, 76.7
// KiB per f32 block).
template <int A> __host__ __device__ constexpr int blocks_per_sm() { return A == BF16 ? 3 : 2; }

// One block per (sequence b, v head h), launched as a programmatic dependent of
// the previous grid on the stream; thread r owns value row r of the state.
// Before waiting for the previous grid the block sets up its barriers (and TMEM)
// and, in the CUDA-core variants, gives L2 hints: its own state (for the blocks
// that become resident while the previous grid drains) and the rows of the unit
// one wave of resident blocks later. Everything the block reads is read after
// the wait (a hint only uses a slot index that may still change). Then the
// conv's loads, the conv_state rows and thread 0's four TMA copies of the state
// (after its conv for T = 3, 4), and per block:
//   - the conv + SiLU of the unit's q, k and v heads for the T draft rows (rows
//     t..t+3 of conv_state ++ x feed token t) and the L2 norms of q and k; q, k and
//     v are kept in f32, unrounded (only the optional post-conv copy is rounded to
//     the activation dtype);
//   - the dot products k_t.k_s (s < t), q_t.k_s (s <= t) and the table
//     b_t r(t,s) (k_t.k_s), r(t,s) (q_t.k_s), g_t, b_t g_t, b_t, with
//     r(t,s) = a_{s+1} ... a_t and g_t = a_0 ... a_t;
//   - the 2T products S0 k_t, S0 q_t of every value row;
//   - deltas, outputs and the z-gated RMSNorm of every draft token.
// Two variants of the products:
//   - CUDA cores (T <= 4, and f32 activations): thread r reads its swizzled f32
//     row with the step kernel's rounding; the dot products are warp dot
//     products with the step kernel's rounding for T <= 2 and 8-lane group dot
//     products (four pairs per warp at once) for T >= 3;
//   - tensor core (TC: bf16 activations, T >= 5): one tcgen05 kind::tf32 product
//     S0 [k_0..k_7 ; q_0..q_7]^T (M = 128, N = 16, K = 128) straight from the TMA
//     boxes, the state and k, q read as tf32; the dot products by 8-lane groups
//     on the CUDA cores, with the table, before the state has arrived (a Gram
//     product on the tensor core after the state wait was 7 % slower at T = 5).
// NT > 0: the number of draft tokens as a compile-time constant (CUDA-core
// variants; keeps the unrolled code small); NT = 0: read from the arguments.
template <int A, bool TC, int NT>
__global__ void __launch_bounds__(VT, blocks_per_sm<A>())
    verify_kernel(StepArgs p, const __grid_constant__ CUtensorMap smap, int ahead) {
  pdl_launch_dependents();
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = NT > 0 ? NT : p.T;
  const int Hk = p.Hk, Hv = p.Hv, G = Hv / Hk, C = (2 * Hk + Hv) * D;
  const int b = blockIdx.x / Hv, h = blockIdx.x % Hv, hq = h / G;

  uint8_t* QK = smem;                                     // q, k; then the outputs
  uint8_t* SR = smem + qk_region<A, TC>();                // the state
  uint8_t* VS = SR + S_BYTES;                             // v rows (CUDA-core variants)
  float* tb = reinterpret_cast<float*>(VS + vs_bytes<TC, NT>());    // the table
  float* al_s = tb + TAB;                                           // alpha, beta
  float* be_s = al_s + MAXT;
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(be_s + MAXT);      // 8-byte aligned
  uint64_t* tc_bar = s_bar + 1;
  uint32_t* tc_slot = reinterpret_cast<uint32_t*>(s_bar + 3);
  uint32_t* issued = tc_slot + 1;                         // 1 once the products were issued

  if (tid == 0) {
    tc::mbar_init(s_bar, 1);
    *issued = 0u;
    if constexpr (TC) {
      tc::mbar_init(tc_bar, 1);
    }
    tc::fence_mbar_init();
  } else if (!TC && warp == 3) {
    // L2 hints (CUDA-core variants; warp 3 has no conv item): this unit's state,
    // and the rows of the unit one wave of resident blocks later, so that its
    // small loads hit L2. The tensor-core variant (T >= 5) runs 3-4 % faster
    // without them.
    if (lane < 4) hint_state(p, &smap, b * Hv + h, lane);
    const int u2 = (int)blockIdx.x + ahead;
    if (u2 < (int)gridDim.x) {
      hint_rows<A>(p, u2, T, lane);
      hint_rows<A>(p, u2, T, lane + 32);
    }
  }
  if constexpr (TC) {
    if (warp == 1) {
      tc::tmem_alloc(tc_slot, 64);                        // the product: 4 x 16 columns
      tc::tmem_relinquish();
    }
  }

  pdl_wait();                                             // inputs of the previous grid are visible
  const int slot = *reinterpret_cast<const volatile int32_t*>(p.slot_idx + b);
  int fail = 0;                                           // 1: before the product, 2: the product

  // Every load that does not depend on the slot goes in flight before the slot
  // is used (b < B, so each of these addresses is in bounds whatever the slot
  // holds): the gates, the z rows and norm_w of the epilogue, the taps and the
  // draft rows of the conv. Then the conv_state rows and the TMA copy of the
  // state, which need the slot.
  const int et = tid >> 4, el16 = tid & 15;
  Raw8<A> zr;
  float nwr[8];
  if (et < T) raw_load<A>(p.z, (((int64_t)b * T + et) * Hv + h) * D + el16 * 8, zr);
  else raw_zero<A>(zr);
  load8<F32>(p.norm_w, el16 * 8, nwr);
  float ga = 0.f, gb = 0.f;
  if (tid < T) {
    const int64_t gi = ((int64_t)b * T + tid) * Hv + h;
    ga = load_gate(p.alpha, gi, p.gate_bf16);
    gb = load_gate(p.beta, gi, p.gate_bf16);
  }

  // ---- post-conv activations, f32 (unrounded; only the post-conv copy is
  // rounded to the activation dtype). Two layouts:
  //   CUDA-core variants up to 4 draft tokens: item (part, head, l16) = thread:
  //     8 channels of head `head` (0 q, 1 k, 2 v) for the IT tokens IT part ..
  //     IT part + IT - 1 (at most 96 items); 16-lane groups share (part, head);
  //     v rows go to VS as f32;
  //   the others (v in registers): q and k: warp w takes tokens w + 4 and w, lanes
  //     0..15 the q head and 16..31 the k head; v: thread r convolves channel r of
  //     the v head for every draft token and keeps v_t[r] in its registers.
  // Tokens 0..2 read conv_state rows, which wait for the slot index; in the
  // register layout every thread convolves its tokens that read draft rows only
  // first (tokens 3.. in the v loop, token w + 4 in the q/k pairs), so that those
  // rows' latency hides behind that work.
  constexpr bool VREG = v_in_regs<TC, NT>();
  // tokens per item: 2 at T = 3, 4 (96 items in place of 48, half the serial
  // work each), else 4; 2 in the register layout
  constexpr int IT = VREG ? 2 : ((NT == 3 || NT == 4) ? 2 : 4);
  float vr[MAXT];                                         // register layout: v_t[r]
  const int64_t xb = (int64_t)b * T * C;
  const bool write_qk = p.postconv && (h % G) == 0;       // one v head of the group writes q, k
  int l16, head, t0;
  bool grp;                                               // a q/k (or q/k/v) item: uniform per 16 lanes
  if constexpr (VREG) {
    grp = warp < (T < 4 ? T : 4);
    l16 = lane & 15; head = lane >> 4; t0 = warp;
  } else {
    grp = tid < (T + IT - 1) / IT * 3 * 16;
    l16 = tid & 15; head = (tid >> 4) % 3; t0 = IT * ((tid >> 4) / 3);
  }
  const int c = (head == 0 ? hq * D : head == 1 ? (Hk + hq) * D : (2 * Hk + h) * D) + l16 * 8;
  // conv rows held per thread: the four rows of each of the two tokens (register
  // layout), else the item's IT + 3 consecutive rows; prow(k) = the row of slot k
  // in the sequence (3 conv_state rows, then the T draft rows)
  constexpr int NR = VREG ? 8 : IT + 3;
  auto prow = [&](int k) { return VREG ? (k < 4 ? t0 + 4 + k : t0 + k - 4) : t0 + k; };
  Raw8<A> wr[4], rw[NR];
#pragma unroll
  for (int j = 0; j < NR; ++j) raw_zero<A>(rw[j]);
  if (grp) {
#pragma unroll
    for (int q = 0; q < 4; ++q) raw_load<A>(p.conv_w, (int64_t)c * KW + 8 * q, wr[q]);
#pragma unroll
    for (int j = 0; j < NR; ++j) {
      const int idx = prow(j);
      if (idx >= KS && idx - KS < T) raw_load<A>(p.x, xb + (int64_t)(idx - KS) * C + c, rw[j]);
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) raw_zero<A>(wr[q]);
  }
  const int cv = (2 * Hk + h) * D + tid;                  // register layout: v channel r
  // register layout: the v channel's taps and rows as raw bits, widened at the v
  // conv, so that the conv_state loads and the state copy are not held up
  uint4 w4r = make_uint4(0u, 0u, 0u, 0u);
  uint32_t colr[MAXT + KS];
  if constexpr (VREG) {
    if constexpr (A == BF16) {
      const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p.conv_w) + (int64_t)cv * KW);
      w4r.x = u.x; w4r.y = u.y;
    } else {
      w4r = *reinterpret_cast<const uint4*>(static_cast<const float*>(p.conv_w) + (int64_t)cv * KW);
    }
#pragma unroll
    for (int j = KS; j < MAXT + KS; ++j) colr[j] = j - KS < T ? load1_bits<A>(p.x, xb + (int64_t)(j - KS) * C + cv) : 0u;
  }

  const bool valid = slot >= 0 && slot < p.n_slots;
  if (slot >= p.n_slots && tid == 0 && h == 0) report(p.dev_err, GDN_DEVERR_SLOT);

  // Thread 0 (which initialised the barrier) starts the TMA copies of the state
  // after its conv_state loads, or, for the 2-token items at T = 3, 4, after its
  // conv: the small loads the conv waits on go first (a state copy issued before
  // them delayed them and made every window slower, by up to 23 %).
  constexpr bool STATE_AFTER_CONV = !TC && (NT == 3 || NT == 4);
  auto start_state_copy = [&]() {
    if (tid == 0) {
      tc::mbar_arrive_expect_tx(s_bar, S_BYTES);
#pragma unroll
      for (int bx = 0; bx < 4; ++bx) tma_load_2d(SR + bx * 16384, &smap, 32 * bx, (slot * Hv + h) * D, s_bar);
    }
  };
  if (valid) {
    const int64_t cs = (int64_t)slot * KS * C;
    if (grp) {                                            // the conv_state rows of the item
#pragma unroll
      for (int j = 0; j < NR; ++j)
        if (prow(j) < KS) raw_load<A>(p.conv_state, cs + (int64_t)prow(j) * C + c, rw[j]);
    }
    if constexpr (VREG) {
#pragma unroll
      for (int j = 0; j < KS; ++j) colr[j] = load1_bits<A>(p.conv_state, cs + (int64_t)j * C + cv);
    }
    if constexpr (!STATE_AFTER_CONV) start_state_copy();
    float2 w[4][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float t8[8];
      raw_unpack<A>(wr[q], t8);
#pragma unroll
      for (int j = 0; j < 4; ++j) w[q][j] = make_float2(t8[j], t8[4 + j]);
    }
    if (!VREG || grp) {                                   // uniform per warp
#pragma unroll
      for (int uu = 0; uu < IT; ++uu) {
        const int t = VREG ? (uu == 0 ? t0 + 4 : t0) : t0 + uu;
        const int k0 = VREG ? 4 * uu : uu;                // the token's first row slot
        const bool live = grp && t < T;
        float v[8];
        if (live) {
          float r0[8], r1[8], r2[8], r3[8];
          raw_unpack<A>(rw[k0], r0);
          raw_unpack<A>(rw[k0 + 1], r1);
          raw_unpack<A>(rw[k0 + 2], r2);
          raw_unpack<A>(rw[k0 + 3], r3);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 a = silu2(conv4x2<A>(w[q][0], w[q][1], w[q][2], w[q][3], make_float2(r0[2 * q], r0[2 * q + 1]),
                                              make_float2(r1[2 * q], r1[2 * q + 1]), make_float2(r2[2 * q], r2[2 * q + 1]),
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
          const float rr = inv_norm(ss, p.eps);
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = __fmul_rn(v[j], rr);
        }
        if (live) {
          if (p.postconv && (head == 2 || write_qk)) store8<A>(p.postconv, xb + (int64_t)t * C + c, v);
          if (head == 2) store8<F32>(VS, (int64_t)t * D + l16 * 8, v);
          else put_act8<A, TC>(QK, head ^ 1, t, l16 * 8, v);   // k rows 0..7, q rows 8..15
        }
      }
    }
    if constexpr (VREG) {
      float w4[4], col[MAXT + KS];
      if constexpr (A == BF16) {
        w4[0] = __uint_as_float(w4r.x << 16); w4[1] = __uint_as_float(w4r.x & 0xffff0000u);
        w4[2] = __uint_as_float(w4r.y << 16); w4[3] = __uint_as_float(w4r.y & 0xffff0000u);
      } else {
        w4[0] = __uint_as_float(w4r.x); w4[1] = __uint_as_float(w4r.y);
        w4[2] = __uint_as_float(w4r.z); w4[3] = __uint_as_float(w4r.w);
      }
#pragma unroll
      for (int j = 0; j < MAXT + KS; ++j) col[j] = bits_to_f<A>(colr[j]);
#pragma unroll
      for (int k = 0; k < MAXT; ++k) {                    // tokens 3 .. 7, then 0 .. 2
        const int t = (k + KS) % MAXT;
        vr[t] = t < T ? silu(conv4(w4, col[t], col[t + 1], col[t + 2], col[t + 3])) : 0.f;
        if (p.postconv && t < T) store1<A>(p.postconv, xb + (int64_t)t * C + cv, vr[t]);
      }
    }
    if constexpr (TC) {                                   // rows of absent tokens are zero operands
      for (int e = tid; e < 16 * (D / 4); e += VT) {
        const int row = e >> 5, kc = e & 31;
        if ((row & 7) >= T) *reinterpret_cast<float4*>(QK + bsw_off(row, 4 * kc)) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if constexpr (STATE_AFTER_CONV) start_state_copy();
    if (tid < T) {                                       // raw projections: the gate step
      al_s[tid] = p.raw_gates ? gate_alpha(ga) : ga;
      be_s[tid] = p.raw_gates ? gate_beta(gb) : gb;
    }
  }

  if constexpr (TC) tc::fence_async_smem();               // the operand rows -> tensor core
  if constexpr (TC) tc::fence_before_sync();
  __syncthreads();                                        // also: barriers and TMEM address visible
  if constexpr (TC) tc::fence_after_sync();
  const uint32_t tbase = TC ? *tc_slot : 0u;

  do {                                                    // once; left early on a failed wait
    if (!valid) break;                                    // padding entry or bad slot: no outputs
    bool ok = true;
    // ---- dot products, in the order t = 0, 1, ...: (k_t.k_s, s < t) then
    // (q_t.k_s, s <= t); the pairs of the first T tokens are the first T^2. On
    // the CUDA cores in every variant, formed (with the table below) while the
    // state is still arriving.
    if constexpr (NT >= 3 || TC) {
      // T >= 3: an 8-lane group per pair (lane holds 16 columns, a product and
      // 15 fused multiply-adds, then an xor butterfly 4, 2, 1), four pairs per
      // warp at once: the T^2 pairs in T^2 / 16 rounds instead of T^2 / 4
      // (these outputs are held to the oracle's tolerance, not to the step
      // kernel's bits, which only T = 1 shares)
      const int sub = lane & 7;
#pragma unroll 1
      for (int i0 = 4 * warp; i0 < T * T; i0 += VT / 8) {
        const int i = i0 + (lane >> 3);
        const bool live = i < T * T;
        const int ii = live ? i : 0;
        const int t = (ii >= 1) + (ii >= 4) + (ii >= 9) + (ii >= 16) + (ii >= 25) + (ii >= 36) + (ii >= 49);
        const int j = ii - t * t, which = j >= t, s = which ? j - t : j;
        float d = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float4 x = act4<A, TC>(QK, which, t, sub + 8 * c);
          const float4 y = act4<A, TC>(QK, 0, s, sub + 8 * c);
          d = c == 0 ? __fmul_rn(x.x, y.x) : __fmaf_rn(x.x, y.x, d);
          d = __fmaf_rn(x.y, y.y, d);
          d = __fmaf_rn(x.z, y.z, d);
          d = __fmaf_rn(x.w, y.w, d);
        }
#pragma unroll
        for (int m = 4; m >= 1; m >>= 1) d = __fadd_rn(d, __shfl_xor_sync(0xffffffffu, d, m));
        if (live && sub == 0) tb[(which ? TAB_OC : TAB_A) + t * MAXT + s] = d;
      }
    } else {
      // T <= 2: warp w takes the pairs w, w + 4, ...; lane l holds columns
      // 4l..4l+3 (a product and three fused multiply-adds), then an xor butterfly
      // 16, 8, 4, 2, 1: the step kernel's warp dot product
#pragma unroll 1
      for (int i = warp; i < T * T; i += VT / 32) {
        const int t = (i >= 1) + (i >= 4) + (i >= 9) + (i >= 16) + (i >= 25) + (i >= 36) + (i >= 49);
        const int j = i - t * t, which = j >= t, s = which ? j - t : j;
        const float4 x = act4<A, TC>(QK, which, t, lane);
        const float4 y = act4<A, TC>(QK, 0, s, lane);
        float d = __fmul_rn(x.x, y.x);
        d = __fmaf_rn(x.y, y.y, d);
        d = __fmaf_rn(x.z, y.z, d);
        d = __fmaf_rn(x.w, y.w, d);
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) d = __fadd_rn(d, __shfl_xor_sync(0xffffffffu, d, m));
        if (lane == 0) tb[(which ? TAB_OC : TAB_A) + t * MAXT + s] = d;
      }
    }
    if (__syncthreads_or(!ok)) { fail = 1; break; }     // also: the dot products are in

    // ---- the table, one entry per thread (which, t, s), from the dot products in
    // place; products in ascending order
    {
      const int which = tid >> 6, t = (tid >> 3) & 7, s = tid & 7;
      if (t < T && (which == 0 ? s < t : s <= t)) {
        float rr = 1.f;
        for (int w = s + 1; w <= t; ++w) rr = __fmul_rn(rr, al_s[w]);
        const float bt = be_s[t];
        if (which == 0) {
          tb[TAB_A + t * MAXT + s] = __fmul_rn(__fmul_rn(bt, rr), tb[TAB_A + t * MAXT + s]);
        } else {
          tb[TAB_OC + t * MAXT + s] = __fmul_rn(rr, tb[TAB_OC + t * MAXT + s]);
          if (s == 0) {
            float gt = al_s[0];
            for (int w = 1; w <= t; ++w) gt = __fmul_rn(gt, al_s[w]);
            tb[TAB_G + t] = gt;
            tb[TAB_BG + t] = __fmul_rn(bt, gt);
            tb[TAB_B + t] = bt;
          }
        }
      }
    }

    // ---- the products
    const int r = tid;                                    // value row
    float sk[MAXT], sq[MAXT];
    if constexpr (TC) {
      // thread 0 waits for the state and issues the state product S0 [k ; q]^T
      // (M = 128, N = 16, K = 128, tf32); four independent accumulators, one per
      // 32-column block of K, keep the accumulation chains short and are summed
      // on the CUDA cores. The dot products and the table were formed on the CUDA
      // cores while the state was still arriving.
      bool ok0 = true;
      if (tid == 0) {
        const uint32_t bq = tc::smem_u32(QK), sa = tc::smem_u32(SR);
        const uint32_t id = tc::idesc_tf32_f32(128, 16);
        ok0 = tc::mbar_wait(s_bar, 0, 1u << 24);
        if (ok0) {
          tc::fence_after_sync();
#pragma unroll 1
          for (int ks = 0; ks < 16; ++ks)
            tc::mma_tf32(tbase + 16 * (ks & 3), smem_desc_sw128(sa + (ks >> 2) * 16384 + (ks & 3) * 32),
                         smem_desc_sw128(bq + (ks >> 2) * 2048 + (ks & 3) * 32), id, ks > 3);
          tc::mma_commit(tc_bar);
          *issued = 1u;
        }
      }
      if (__syncthreads_or(!ok0)) { fail = 1; break; }    // the state wait gave up
      ok = tc::mbar_wait(tc_bar, 0, 1u << 24);
      tc::fence_after_sync();
      if (__syncthreads_or(!ok)) { fail = 2; break; }     // also: the table is complete
      float acc[16];
      sum4_ld16(tbase + ((uint32_t)(32 * warp) << 16), acc);
#pragma unroll
      for (int t = 0; t < MAXT; ++t) { sk[t] = acc[t]; sq[t] = acc[8 + t]; }
    } else {
      ok = tc::mbar_wait(s_bar, 0, 1u << 24);
      if (__syncthreads_or(!ok)) { fail = 1; break; }     // also: the table is complete
      // row r with the step kernel's rounding: four partial sums over the chunks
      // j = 4m + cg (m ascending), then (p0 + p1) + (p2 + p3)
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
            const float4 k = act4<A, TC>(QK, 0, t, j);
            float a = pk[t][cg];
            a = __fmaf_rn(s4.x, k.x, a); a = __fmaf_rn(s4.y, k.y, a);
            a = __fmaf_rn(s4.z, k.z, a); a = __fmaf_rn(s4.w, k.w, a);
            pk[t][cg] = a;
            const float4 q = act4<A, TC>(QK, 1, t, j);
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
    if constexpr (TC) tc::fence_before_sync();
    __syncthreads();                                      // q and k are no longer needed

    // ---- deltas and outputs of row r (the step kernel's order)
    float o[MAXT];
    {
      float dr[MAXT];
#pragma unroll
      for (int t = 0; t < MAXT; ++t) {
        if (t < T) {
          const float vt = v_in_regs<TC, NT>() ? vr[t] : reinterpret_cast<const float*>(VS)[t * D + r];
          float xx = __fmaf_rn(-tb[TAB_BG + t], sk[t], __fmul_rn(tb[TAB_B + t], vt));
#pragma unroll
          for (int w = 0; w < t; ++w) xx = __fmaf_rn(-tb[TAB_A + t * MAXT + w], dr[w], xx);
          dr[t] = xx;
          float y = __fmul_rn(tb[TAB_G + t], sq[t]);
#pragma unroll
          for (int w = 0; w <= t; ++w) y = __fmaf_rn(tb[TAB_OC + t * MAXT + w], dr[w], y);
          o[t] = __fmul_rn(y, p.q_scale);
        }
      }
    }
    float* o_s = reinterpret_cast<float*>(QK);            // [T][128] f32
#pragma unroll
    for (int t = 0; t < MAXT; ++t)
      if (t < T) o_s[t * D + r] = o[t];
    __syncthreads();

    // ---- z-gated RMSNorm: one 16-lane group per token
    {
      const bool live = et < T;
      float ov[8];
      if (live) {
        const float4 u0 = reinterpret_cast<const float4*>(o_s + et * D)[2 * el16];
        const float4 u1 = reinterpret_cast<const float4*>(o_s + et * D)[2 * el16 + 1];
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
        raw_unpack<A>(zr, zv);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          res[j] = __fmul_rn(__fmul_rn(__fmul_rn(ov[j], rn), nwr[j]), silu_gate(zv[j]));
        store_out8<A>(p.out, ((int64_t)b * T + et) * Hv * D + (int64_t)h * D + el16 * 8, res, p.out_f32);
      }
    }
  } while (false);

  if (fail) {                       // a wait gave up: no outputs for this (sequence, head)
    if (tid == 0) report(p.dev_err, GDN_DEVERR_TIMEOUT);
    tc::mbar_wait(s_bar, 0, 1u << 24);                    // the state copy, if still in flight
    if constexpr (TC) {
      if (*issued) {                                      // set before the failing barrier
        tc::mbar_wait(tc_bar, 0, 1u << 24);               // the state product, if still running
      }
    }
  }
  if constexpr (TC) {
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) tc::tmem_dealloc(tbase, 64);
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
cudaError_t launch_kernel(const StepArgs& a, const CUtensorMap& smap, cudaStream_t stream) {
  auto kern = verify_kernel<A, TC, NT>;
  const int smem = verify_smem<A, TC, NT>();
  cudaError_t e = set_smem_once<verify_kernel<A, TC, NT>>(smem, true);
  if (e != cudaSuccess) return e;
  int n_sm = 0;
  if ((e = sm_count(&n_sm)) != cudaSuccess) return e;
  const int ahead = blocks_per_sm<A>() * n_sm;              // blocks resident at once
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((int64_t)a.B * a.Hv));
  cfg.blockDim = dim3(VT);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, smap, ahead);
}

template <int A>
cudaError_t launch_verify_impl(const StepArgs& a, cudaStream_t stream) {
  CUtensorMap smap;
  cudaError_t e = state_map(a, &smap);
  if (e != cudaSuccess) return e;
  if constexpr (A == BF16) {
    switch (a.T) {
      case 1: return launch_kernel<A, false, 1>(a, smap, stream);
      case 2: return launch_kernel<A, false, 2>(a, smap, stream);
      case 3: return launch_kernel<A, false, 3>(a, smap, stream);
      case 4: return launch_kernel<A, false, 4>(a, smap, stream);
      default: return launch_kernel<A, true, 0>(a, smap, stream);
    }
  } else {
    switch (a.T) {
      case 1: return launch_kernel<A, false, 1>(a, smap, stream);
      case 2: return launch_kernel<A, false, 2>(a, smap, stream);
      case 3: return launch_kernel<A, false, 3>(a, smap, stream);
      case 4: return launch_kernel<A, false, 4>(a, smap, stream);
      case 5: return launch_kernel<A, false, 5>(a, smap, stream);
      case 6: return launch_kernel<A, false, 6>(a, smap, stream);
      case 7: return launch_kernel<A, false, 7>(a, smap, stream);
      case 8: return launch_kernel<A, false, 8>(a, smap, stream);
      default: return cudaErrorInvalidValue;               // T is 1..8 (checked by the API)
    }
  }
}

}  // namespace

// bf16 activations with two or more draft tokens take the tensor-core product;
// T = 1 and f32 activations the CUDA-core rows.
cudaError_t launch_verify_readonly(const StepArgs& a, int act, cudaStream_t stream) {
  return act == GDN_BF16 ? launch_verify_impl<BF16>(a, stream) : launch_verify_impl<F32>(a, stream);
}

}  // namespace gdn
