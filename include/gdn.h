/*
 * gdn.h — C ABI of the Gated DeltaNet token-mixing library for GB300 (sm_103a).
 *
 * The path: width-4 depthwise causal conv1d over packed q|k|v channels with a
 * per-sequence conv_state, SiLU, per-head L2 normalisation of q and k, the
 * gated delta-rule recurrence
 *     S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,   o_t = S_t q_t,
 * and a z-gated RMSNorm of o_t. Three phases use it: varlen prefill, the
 * speculative verify of T = 1..8 draft tokens, and the commit of the accepted
 * prefix of conv_state and recurrent state across all layers.
 *
 * Sources (page title, section):
 *   "perf(gdn): optimize post-conv and causal-conv kernels - #155" — the causal
 *     conv ("Blocker"), the post-conv 128-lane sum of squares then 1/sqrt and the
 *     initial/final conv_state rows of exact chunks ("Merged ...", "New issue #305");
 *     exact causal-conv chunk descriptors ("Before starting").
 *   "Strata PR #3226" — speculative verify over T draft tokens, the output norm,
 *     and the one-call commit of conv_state and state for all layers ("Summary");
 *     the fused gate kernel ("Root Cause & RED / GREEN Verification") and the
 *     forward that commits inside itself ("Problem and result").
 *
 * Entry points: gdn_conv_fwd, gdn_postconv_norm, gdn_delta_prefill,
 * gdn_verify_step (and gdn_verify_step_noalloc), gdn_commit_layers,
 * gdn_verify_step_lazy, gdn_gates; gdn_verify_workspace_bytes and
 * gdn_status_string are helpers.
 *
 * Conventions shared by every entry point
 *   - head_dim d = 128 and conv width 4 are the only supported values.
 *   - C = (2*Hk + Hv) * 128 packed channels [q heads | k heads | v heads]; v head
 *     h reads q/k head h / (Hv/Hk).
 *   - Activations (x, post-conv rows, z, out, conv_w, conv_state) have the dtype
 *     cfg->act: GDN_F32 or GDN_BF16 (out may be f32 instead, cfg->out_f32). The
 *     gates alpha, beta (or raw a, b) have the dtype cfg->gate_dtype. norm_w and
 *     the state S are f32.
 *   - Layouts are row-major: x/qkv [n_tok][C]; conv_w [C][4] (tap 3 multiplies
 *     the current token); conv_state pool [n_slots][3][C] (oldest row first);
 *     state pool [n_slots][Hv][128 value rows][128 key columns] f32;
 *     alpha/beta [tokens][Hv]; z/out [tokens][Hv*128]; norm_w [128].
 *   - All pointers are caller-owned DEVICE memory unless stated. The library
 *     allocates nothing, keeps no state between calls, never synchronises, and
 *     enqueues its kernels on `stream` (a cudaStream_t; NULL = legacy default).
 *   - Every pointer must be 16-byte aligned; leading dimensions are in elements
 *     and must keep rows 16-byte aligned.
 *   - Errors: host-side validation failures return GDN_ERR_INVALID or
 *     GDN_ERR_UNSUPPORTED and enqueue nothing; a failed launch returns
 *     GDN_ERR_CUDA. Bad device-resident indices (a slot >= cfg->n_slots, n_keep
 *     outside [0, T], inconsistent cu_seqlens) skip the affected sequence and OR
 *     a GDN_DEVERR_* bit into *cfg->dev_err when that pointer is non-null. A
 *     negative slot index marks padding: the entry is skipped without error.
 *   - In a call that writes conv_state or state (gdn_conv_fwd, gdn_delta_prefill,
 *     gdn_verify_step with GDN_VERIFY_COMMIT_ALL, gdn_commit_layers,
 *     gdn_verify_step_lazy) the non-negative slot indices must be pairwise
 *     distinct: entries naming the same slot would update it from different
 *     blocks at once, and the result is undefined. Read-only calls may repeat
 *     slots.
 */
#ifndef GDN_H
#define GDN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID = 1,      /* null pointer, bad shape, aliasing, misalignment */
  GDN_ERR_UNSUPPORTED = 2,  /* head_dim != 128, conv_width != 4, unknown dtype */
  GDN_ERR_CUDA = 3          /* a kernel launch failed */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

#define GDN_HEAD_DIM 128
#define GDN_CONV_WIDTH 4
#define GDN_MAX_DRAFT 8
#define GDN_CHUNK 64

/* gdn_config.gates: what the alpha / beta arguments hold */
#define GDN_GATES_ACTIVATED 0     /* the gates alpha_t, beta_t themselves */
#define GDN_GATES_RAW 1           /* raw projections a_t, b_t: each kernel applies the
                                     gate step (see gdn_gates) to the values it reads */

/* verify flags */
#define GDN_VERIFY_COMMIT_ALL 1u  /* accept every draft token: advance conv_state
                                     and state in place (decode) */

/* device error bits */
#define GDN_DEVERR_SLOT 1u        /* slot index >= n_slots */
#define GDN_DEVERR_NKEEP 2u       /* n_keep outside [0, T] */
#define GDN_DEVERR_SEQLENS 4u     /* cu_seqlens decreasing or beyond n_tok */
#define GDN_DEVERR_TIMEOUT 8u     /* a tensor-core completion wait gave up; the
                                     sequence's outputs and state are incomplete */

typedef struct gdn_config {
  int32_t n_qk_heads;   /* Hk >= 1 */
  int32_t n_v_heads;    /* Hv >= 1, a multiple of Hk */
  int32_t head_dim;     /* must be 128 */
  int32_t conv_width;   /* must be 4 */
  int32_t act;          /* gdn_dtype of the activations */
  float eps;            /* epsilon of the q/k L2 norm and of the RMSNorm (inside the root) */
  float q_scale;        /* multiplies o_t; 1.0 gives o_t = S_t q_t */
  int32_t n_slots;      /* slots in the conv_state and state pools */
  uint32_t* dev_err;    /* nullable device word receiving GDN_DEVERR_* bits */
  int32_t gates;        /* GDN_GATES_ACTIVATED (0) or GDN_GATES_RAW: applies to the
                           alpha / beta arguments of gdn_delta_prefill and
                           gdn_verify_step and to the layer views of gdn_commit_layers */
  int32_t gate_dtype;   /* element type of every gate array (alpha, beta, raw a, b, and
                           the outputs of gdn_gates): GDN_F32 (0) or GDN_BF16. A bf16
                           gate is widened exactly to f32 where it is read. */
  int32_t out_f32;      /* 0: out has the activation dtype; 1: out is f32 (the z-gated
                           RMSNorm's result stored without rounding), for
                           gdn_delta_prefill, gdn_verify_step(_noalloc, _lazy) */
} gdn_config;

/* One layer's device views for gdn_commit_layers (the array itself lives in
 * device memory). x, alpha, beta are that layer's verify inputs (raw
 * projections a, b when the config's gates is GDN_GATES_RAW). */
typedef struct gdn_layer_view {
  const void* x;         /* [B][T][C] act */
  const void* alpha;     /* [B][T][Hv] gate_dtype */
  const void* beta;      /* [B][T][Hv] gate_dtype */
  const void* conv_w;    /* [C][4] act */
  void* conv_state;      /* [n_slots][3][C] act, updated in place */
  float* state;          /* [n_slots][Hv][128][128], updated in place */
} gdn_layer_view;

/*
 * gdn_conv_fwd — varlen causal conv1d (width 4) + SiLU (+ q/k L2 norm).
 * Source: "perf(gdn) ... #155" — the causal conv and its exact 64-token chunks
 * aligned to each sequence start; the initial conv_state is read and the final
 * one written by the same thread block (the chunk-0 block), so the read/write
 * race of "New issue #305" cannot occur.
 *
 *   x          [n_tok][ld_x] act; sequence s owns rows cu_seqlens[s]..cu_seqlens[s+1]-1
 *   y          [n_tok][ld_y] act; must not overlap x (other blocks read x halos)
 *   conv_w     [C][4] act
 *   conv_state pool; slot slot_idx[s] is read when has_init[s] (else zeros) and
 *              always receives the last 3 rows of (initial rows ++ x rows of s)
 *   slot_idx   [n_seq] int32, cu_seqlens [n_seq+1] int32, has_init [n_seq] uint8
 *   fuse_norm  1: L2-normalise q and k heads of the SiLU output (f32 math before
 *              the store); 0: store SiLU output only (see gdn_postconv_norm)
 * Every sequence, empty ones included, commits its conv_state.
 */
gdn_status gdn_conv_fwd(const gdn_config* cfg, const void* x, int64_t ld_x, void* y,
                        int64_t ld_y, const void* conv_w, void* conv_state,
                        const int32_t* slot_idx, const int32_t* cu_seqlens,
                        const uint8_t* has_init, int32_t n_seq, int64_t n_tok,
                        int32_t fuse_norm, void* stream);

/*
 * gdn_postconv_norm — per-head L2 norm of the q and k heads of post-conv rows;
 * v channels are copied (converted to out_t).
 * Source: "perf(gdn) ... #155", "Merged ...": 128-lane sum of squares, then
 * 1/sqrt, then scale. The f32 order is fixed: squares of 16 groups of 8
 * contiguous channels folded with strides 4, 2, 1, then the 16 group sums with
 * strides 8, 4, 2, 1; r = 1/sqrt(sum + eps) with correctly rounded sqrt and
 * divide. An f32 -> f32 call is therefore bitwise reproducible.
 *   y_in [n_tok][C] in_t, y_out [n_tok][C] out_t; y_out may equal y_in when
 *   in_t == out_t (in place); partial overlap is invalid.
 */
gdn_status gdn_postconv_norm(const gdn_config* cfg, int32_t in_t, const void* y_in,
                             int32_t out_t, void* y_out, int64_t n_tok, void* stream);

/*
 * gdn_delta_prefill — chunked (WY-form) gated delta rule over varlen sequences,
 * with the z-gated RMSNorm fused into the output.
 * Source: the recurrence S_t = a_t S_{t-1}(I - b_t k_t k_t^T) + b_t v_t k_t^T,
 * o_t = S_t q_t, and "Strata PR #3226" (output norm after the recurrence).
 *   qkv     [n_tok][C] act: post-conv rows (q, k L2-normalised), e.g. from
 *           gdn_conv_fwd(fuse_norm=1)
 *   alpha, beta [n_tok][Hv] gate_dtype: the gates, or the raw a, b when
 *               cfg->gates is GDN_GATES_RAW
 *   z       [n_tok][Hv*128] act
 *   out     [n_tok][Hv*128] act (f32 when cfg->out_f32); out = RMSNorm(o) *
 *           norm_w * silu(z)
 *   norm_w  [128] f32
 *   state   pool: read at slot_idx[s] when has_init[s] (else zero), always
 *           written with the state after the last token of s
 *   chunk   must be GDN_CHUNK (64)
 */
gdn_status gdn_delta_prefill(const gdn_config* cfg, const void* qkv, const void* alpha,
                             const void* beta, const void* z, const float* norm_w, void* out,
                             float* state, const int32_t* slot_idx, const int32_t* cu_seqlens,
                             const uint8_t* has_init, int32_t n_seq, int64_t n_tok,
                             int32_t chunk, void* stream);

/*
 * gdn_verify_workspace_bytes — bytes of device workspace gdn_verify_step needs
 * for B sequences of T draft tokens: 0 for every valid configuration (the
 * verify kernel keeps its intermediate results on chip), -1 for an invalid one.
 * Kept so that callers size the workspace argument from the library. The pages
 * have no counterpart: it is a property of this implementation.
 */
int64_t gdn_verify_workspace_bytes(const gdn_config* cfg, int32_t B, int32_t T);

/*
 * gdn_verify_step — speculative verify of T draft tokens for B sequences of one
 * layer: conv from conv_state (+SiLU, +L2 norm), the recurrence from the current
 * state, and the gated RMSNorm, for every draft token.
 * Source: "Strata PR #3226" ("Summary": verify forward launched once per layer).
 *   x       [B][T][C] act (raw, pre-conv rows of the draft tokens)
 *   alpha, beta [B][T][Hv] gate_dtype (raw a, b when cfg->gates is GDN_GATES_RAW)
 *   z       [B][T][Hv*128] act; norm_w [128] f32
 *   out     [B][T][Hv*128] act (f32 when cfg->out_f32)
 *   The post-conv activations enter the recurrence unrounded (f32): they are
 *   never stored here (only their rounded copy, postconv_out, when asked for).
 *   Products: f32 on the CUDA cores, except bf16 activations with T >= 5, whose
 *   S0 k_t, S0 q_t and k.k, q.k products run on the tensor core in tf32 (10
 *   explicit mantissa bits): their f32 outputs are within 4e-3 * max(1, |exact|)
 *   of the exact value, their bf16 outputs within the bf16 rounding.
 *   slot_idx [B] int32 into both pools
 *   flags   0: conv_state and state are only read;
 *           GDN_VERIFY_COMMIT_ALL: both advance in place by all T tokens,
 *           bitwise equal to this call without the flag followed by
 *           gdn_commit_layers with n_keep = T.
 *   postconv_out  nullable [B][T][C] act: the post-conv activations used
 *   workspace, workspace_bytes  gdn_verify_workspace_bytes(cfg, B, T) bytes of
 *                 caller-owned device memory; that is 0, so both may be NULL / 0
 *                 (a non-NULL pointer is not accessed). GDN_ERR_INVALID for
 *                 workspace_bytes < 0, or NULL with workspace_bytes != 0.
 *   T in 1..GDN_MAX_DRAFT.
 */
gdn_status gdn_verify_step(const gdn_config* cfg, const void* x, const void* conv_w,
                           void* conv_state, float* state, const void* alpha,
                           const void* beta, const void* z, const float* norm_w, void* out,
                           const int32_t* slot_idx, int32_t B, int32_t T, uint32_t flags,
                           void* postconv_out, void* workspace, int64_t workspace_bytes,
                           void* stream);

/*
 * gdn_verify_step_noalloc — the read-only gdn_verify_step (no
 * GDN_VERIFY_COMMIT_ALL) for callers that cannot allocate device memory: code
 * hosted inside a framework or runtime that owns every device allocation and
 * gives its plugins no allocator, services that run under a fixed device-memory
 * budget, and loops that must not call cudaMalloc/cudaFree because those calls
 * can synchronise the device. The pages have no counterpart; it exists only for
 * such callers.
 *
 * Arguments are those of gdn_verify_step, minus flags, workspace and
 * workspace_bytes; conv_state and state are only read; errors as for
 * gdn_verify_step. It allocates nothing and frees nothing, and uses no memory
 * of its own: the verify kernel needs no workspace, so this is gdn_verify_step
 * with that guarantee stated. Calls may overlap on the GPU (they share nothing
 * but their arguments).
 */
gdn_status gdn_verify_step_noalloc(const gdn_config* cfg, const void* x, const void* conv_w,
                                   const void* conv_state, const float* state, const void* alpha,
                                   const void* beta, const void* z, const float* norm_w, void* out,
                                   const int32_t* slot_idx, int32_t B, int32_t T, void* postconv_out,
                                   void* stream);

/*
 * gdn_commit_layers — commit the accepted prefix of a verify window in every
 * layer in one call: for each layer l and batch entry b with 0 < n = n_keep[b]
 * <= T, conv_state <- last 3 rows of (conv_state ++ x[b, 0:n]) and state <- the
 * state after the first n draft tokens, recomputed exactly as gdn_verify_step
 * computes them. n_keep[b] == 0 leaves slot b untouched in every layer.
 * Source: "Strata PR #3226", "Summary" item 1 (batched commit across layers).
 *   layers  DEVICE array [L] of gdn_layer_view
 *   slot_idx, n_keep [B] int32 (device), shared by all layers
 * The result for a (layer, slot, n_keep) is bitwise independent of L, B and of
 * how layers are grouped into calls.
 */
gdn_status gdn_commit_layers(const gdn_config* cfg, const gdn_layer_view* layers, int32_t L,
                             const int32_t* slot_idx, const int32_t* n_keep, int32_t B,
                             int32_t T, void* stream);

/*
 * gdn_verify_step_lazy — the verify of T new draft tokens with the commit of the
 * previous window's accepted prefix folded in, for one layer.
 * Source: "Strata PR #3226" — "Summary": the verify forward launched once per
 * layer and the batched commit of the accepted prefix of conv_state and state;
 * "Problem and result": a forward variant that commits inside the forward
 * (commit_state = true), tested bitwise against the forward without it followed
 * by the separate commit. Here the commit of one window rides on the next
 * window's forward.
 *
 * Equivalent to gdn_commit_layers over this one layer with (prev_x, prev_alpha,
 * prev_beta, prev_n_keep, prev_T), followed by gdn_verify_step (read-only) of
 * (x, alpha, beta, T): conv_state and state leave the call bitwise equal to that
 * commit (same instructions), and nothing of the new drafts is written back, so
 * the next window passes this window's inputs and accepted prefixes as prev_*.
 * The state is read from HBM once per call, not twice (verify, then commit).
 * The outputs come from the step kernel's CUDA-core products on the committed
 * state (bitwise equal to decode's arithmetic, within the bf16 / f32
 * tolerances of gdn_verify_step's).
 *
 *   prev_x        [B][prev_T][C] act: the previous window's draft rows of this layer
 *   prev_alpha, prev_beta  [B][prev_T][Hv] gate_dtype (raw a, b in GDN_GATES_RAW mode)
 *   prev_n_keep   [B] int32 in [0, prev_T]: accepted tokens of the previous window
 *                 (0: nothing to commit for that sequence)
 *   the other arguments as gdn_verify_step's (without flags and workspace); row b
 *   is the same sequence (slot_idx[b]) in both windows.
 * Errors: GDN_ERR_INVALID for null pointers, T or prev_T outside 1..GDN_MAX_DRAFT,
 * misalignment, out overlapping x, z or prev_x. A prev_n_keep outside
 * [0, prev_T] sets GDN_DEVERR_NKEEP and skips that sequence (nothing written).
 */
gdn_status gdn_verify_step_lazy(const gdn_config* cfg, const void* prev_x, const void* prev_alpha,
                                const void* prev_beta, const int32_t* prev_n_keep, int32_t prev_T,
                                const void* x, const void* conv_w, void* conv_state, float* state,
                                const void* alpha, const void* beta, const void* z,
                                const float* norm_w, void* out, const int32_t* slot_idx, int32_t B,
                                int32_t T, void* postconv_out, void* stream);

/*
 * gdn_gates — the gate step: alpha = exp(-softplus(a)), beta = sigmoid(b),
 * softplus(a) = log(1 + e^a), elementwise over n_tok rows of Hv values.
 * Source: "Strata PR #3226", "Root Cause & RED / GREEN Verification" — a fused
 * gate kernel and its multi-token form, tested bitwise against each other; the
 * pages print no formula, and the form here is the one that defines the gates
 * of the synthetic workloads. In GDN_GATES_RAW mode the prefill, verify and
 * commit kernels apply the same device function to the raw values they read,
 * so their results are bitwise those of gdn_gates followed by the same call in
 * GDN_GATES_ACTIVATED mode.
 *
 *   a, b          [n_tok][Hv] raw projections (device), cfg->gate_dtype
 *   alpha, beta   [n_tok][Hv] results (device, caller-owned), cfg->gate_dtype
 *                 (bf16 results are rounded to nearest even from the f32 values);
 *                 alpha may be a and beta may be b (in place), other overlaps are
 *                 invalid
 *   cfg->gates is not read (the call always applies the gate step).
 * Accuracy: CUDA's expf / log1pf and a correctly rounded divide, within a few
 * ulp of the exact gates (alpha's relative error grows with softplus(a)).
 * Errors: GDN_ERR_INVALID for null pointers (n_tok > 0), n_tok < 0 or bad
 * overlaps; GDN_ERR_CUDA if the launch fails. n_tok == 0 enqueues nothing.
 */
gdn_status gdn_gates(const gdn_config* cfg, const void* a, const void* b, void* alpha,
                     void* beta, int64_t n_tok, void* stream);

/* Static description of a status code (never NULL; "unknown status" for a value
 * outside gdn_status; the string is owned by the library). The pages have no
 * counterpart: it exists for callers' error messages. */
const char* gdn_status_string(gdn_status s);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
