// C ABI of the GDN library: host-side validation, then kernel launches on the
// caller's stream. Nothing here allocates, synchronises or keeps state.
#include <cstdint>
#include <cstring>

#include "launch.h"


namespace {

constexpr int MAX_GROUP = 16;   // v heads per q/k head supported by the step kernels

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t esize(int dt) { return dt == GDN_BF16 ? 2 : 4; }

gdn_status check_cfg(const gdn_config* cfg) {
  if (!cfg) return GDN_ERR_INVALID;
  if (cfg->head_dim != GDN_HEAD_DIM || cfg->conv_width != GDN_CONV_WIDTH) return GDN_ERR_UNSUPPORTED;
  if (cfg->act != GDN_F32 && cfg->act != GDN_BF16) return GDN_ERR_UNSUPPORTED;
  if (cfg->n_qk_heads < 1 || cfg->n_v_heads < 1 || cfg->n_v_heads % cfg->n_qk_heads != 0)
    return GDN_ERR_INVALID;
  if (cfg->n_v_heads / cfg->n_qk_heads > MAX_GROUP) return GDN_ERR_UNSUPPORTED;
  if (cfg->n_slots < 1) return GDN_ERR_INVALID;
  if (!(cfg->eps >= 0.f)) return GDN_ERR_INVALID;
  if (cfg->dev_err && (reinterpret_cast<uintptr_t>(cfg->dev_err) & 3u)) return GDN_ERR_INVALID;
  if (cfg->gates != GDN_GATES_ACTIVATED && cfg->gates != GDN_GATES_RAW) return GDN_ERR_INVALID;
  if (cfg->gate_dtype != GDN_F32 && cfg->gate_dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
  if (cfg->out_f32 != 0 && cfg->out_f32 != 1) return GDN_ERR_INVALID;
  return GDN_OK;
}

// Bytes of one element of `out`.
size_t out_esize(const gdn_config* cfg) { return cfg->out_f32 ? 4 : (cfg->act == GDN_BF16 ? 2 : 4); }

// The arguments shared by the step launches (verify, decode, commit, lazy).
gdn::StepArgs step_args(const gdn_config* cfg, int B, int T) {
  gdn::StepArgs a{};
  a.B = B;
  a.T = T;
  a.Hk = cfg->n_qk_heads;
  a.Hv = cfg->n_v_heads;
  a.n_slots = cfg->n_slots;
  a.eps = cfg->eps;
  a.q_scale = cfg->q_scale;
  a.dev_err = cfg->dev_err;
  a.raw_gates = cfg->gates == GDN_GATES_RAW;
  a.gate_bf16 = cfg->gate_dtype == GDN_BF16;
  a.out_f32 = cfg->out_f32;
  return a;
}

int64_t channels(const gdn_config* cfg) {
  return (int64_t)(2 * cfg->n_qk_heads + cfg->n_v_heads) * GDN_HEAD_DIM;
}

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na && nb && x < y + nb && y < x + na;
}

gdn_status from_cuda(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

}  // namespace

extern "C" {

const char* gdn_status_string(gdn_status s) {
  switch (s) {
    case GDN_OK: return "ok";
    case GDN_ERR_INVALID: return "invalid argument";
    case GDN_ERR_UNSUPPORTED: return "unsupported configuration";
    case GDN_ERR_CUDA: return "CUDA launch failed";
  }
  return "unknown status";
}

gdn_status gdn_conv_fwd(const gdn_config* cfg, const void* x, int64_t ld_x, void* y,
                        int64_t ld_y, const void* conv_w, void* conv_state,
                        const int32_t* slot_idx, const int32_t* cu_seqlens,
                        const uint8_t* has_init, int32_t n_seq, int64_t n_tok,
                        int32_t fuse_norm, void* stream) {
  gdn_status st = check_cfg(cfg);
  if (st != GDN_OK) return st;
  if (n_seq < 0 || n_tok < 0) return GDN_ERR_INVALID;
  if (n_seq == 0) return GDN_OK;
  if (!x || !y || !conv_w || !conv_state || !slot_idx || !cu_seqlens || !has_init)
    return GDN_ERR_INVALID;
  const int64_t C = channels(cfg);
  if (ld_x < C || ld_y < C || ld_x % 8 || ld_y % 8) return GDN_ERR_INVALID;
  if (!aligned16(x) || !aligned16(y) || !aligned16(conv_w) || !aligned16(conv_state))
    return GDN_ERR_INVALID;
  const size_t es = esize(cfg->act);
  if (overlap(x, (size_t)n_tok * ld_x * es, y, (size_t)n_tok * ld_y * es)) return GDN_ERR_INVALID;
  const int64_t blocks = (n_tok + GDN_CHUNK - 1) / GDN_CHUNK + n_seq;
  if (blocks > 0x7fffffff) return GDN_ERR_INVALID;
  return from_cuda(gdn::launch_conv_fwd(*cfg, x, ld_x, y, ld_y, conv_w, conv_state, slot_idx,
                                        cu_seqlens, has_init, n_seq, n_tok, fuse_norm != 0,
                                        static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_postconv_norm(const gdn_config* cfg, int32_t in_t, const void* y_in,
                             int32_t out_t, void* y_out, int64_t n_tok, void* stream) {
  gdn_status st = check_cfg(cfg);
  if (st != GDN_OK) return st;
  if ((in_t != GDN_F32 && in_t != GDN_BF16) || (out_t != GDN_F32 && out_t != GDN_BF16))
    return GDN_ERR_UNSUPPORTED;
  if (n_tok < 0) return GDN_ERR_INVALID;
  if (n_tok == 0) return GDN_OK;
  if (!y_in || !y_out || !aligned16(y_in) || !aligned16(y_out)) return GDN_ERR_INVALID;
  const int64_t C = channels(cfg);
  const size_t ni = (size_t)n_tok * C * esize(in_t), no = (size_t)n_tok * C * esize(out_t);
  const bool same = y_in == y_out && in_t == out_t;
  if (!same && overlap(y_in, ni, y_out, no)) return GDN_ERR_INVALID;
  int n_sm = 0;
  if (gdn::sm_count(&n_sm) != cudaSuccess) return GDN_ERR_CUDA;
  return from_cuda(gdn::launch_postconv_norm(*cfg, in_t, y_in, out_t, y_out, n_tok, n_sm,
                                             static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_delta_prefill(const gdn_config* cfg, const void* qkv, const void* alpha,
                             const void* beta, const void* z, const float* norm_w, void* out,
                             float* state, const int32_t* slot_idx, const int32_t* cu_seqlens,
                             const uint8_t* has_init, int32_t n_seq, int64_t n_tok,
                             int32_t chunk, void* stream) {
  gdn_status st = check_cfg(cfg);
  if (st != GDN_OK) return st;
  if (chunk != GDN_CHUNK) return GDN_ERR_UNSUPPORTED;
  if (n_seq < 0 || n_tok < 0) return GDN_ERR_INVALID;
  if (n_seq == 0) return GDN_OK;
  if (!qkv || !alpha || !beta || !z || !norm_w || !out || !state || !slot_idx || !cu_seqlens ||
      !has_init)
    return GDN_ERR_INVALID;
  if (!aligned16(qkv) || !aligned16(z) || !aligned16(out) || !aligned16(state)) return GDN_ERR_INVALID;
  const size_t es = esize(cfg->act), eo = out_esize(cfg);
  const size_t HvD = (size_t)cfg->n_v_heads * GDN_HEAD_DIM;
  if (overlap(out, (size_t)n_tok * HvD * eo, qkv, (size_t)n_tok * channels(cfg) * es) ||
      overlap(out, (size_t)n_tok * HvD * eo, z, (size_t)n_tok * HvD * es))
    return GDN_ERR_INVALID;
  if (n_seq > 65535) return GDN_ERR_UNSUPPORTED;
  gdn::PrefillArgs a{};
  a.qkv = qkv; a.alpha = alpha; a.beta = beta; a.z = z; a.norm_w = norm_w; a.out = out;
  a.state = state; a.slot_idx = slot_idx; a.cu = cu_seqlens; a.has_init = has_init;
  a.n_seq = n_seq; a.Hk = cfg->n_qk_heads; a.Hv = cfg->n_v_heads; a.n_slots = cfg->n_slots;
  a.n_tok = n_tok; a.eps = cfg->eps; a.q_scale = cfg->q_scale; a.dev_err = cfg->dev_err;
  a.raw_gates = cfg->gates == GDN_GATES_RAW;
  a.gate_bf16 = cfg->gate_dtype == GDN_BF16;
  a.out_f32 = cfg->out_f32;
  return from_cuda(gdn::launch_prefill(a, cfg->act, static_cast<cudaStream_t>(stream)));
}

int64_t gdn_verify_workspace_bytes(const gdn_config* cfg, int32_t B, int32_t T) {
  if (check_cfg(cfg) != GDN_OK || B < 0 || T < 1 || T > GDN_MAX_DRAFT) return -1;
  return 0;                                   // the verify kernel needs no workspace
}

gdn_status gdn_verify_step(const gdn_config* cfg, const void* x, const void* conv_w,
                           void* conv_state, float* state, const void* alpha,
                           const void* beta, const void* z, const float* norm_w, void* out,
                           const int32_t* slot_idx, int32_t B, int32_t T, uint32_t flags,
                           void* postconv_out, void* workspace, int64_t workspace_bytes,
                           void* stream) {
  gdn_status st = check_cfg(cfg);
  if (st != GDN_OK) return st;
  if (B < 0 || T < 1 || T > GDN_MAX_DRAFT) return GDN_ERR_INVALID;
  if (flags & ~GDN_VERIFY_COMMIT_ALL) return GDN_ERR_INVALID;
  if (B == 0) return GDN_OK;
  if (B > 65535) return GDN_ERR_UNSUPPORTED;
  if (!x || !conv_w || !conv_state || !state || !alpha || !beta || !z || !norm_w || !out ||
      !slot_idx)
    return GDN_ERR_INVALID;
  if (!aligned16(x) || !aligned16(conv_w) || !aligned16(conv_state) || !aligned16(state) ||
      !aligned16(z) || !aligned16(out) || !aligned16(norm_w) ||
      (postconv_out && !aligned16(postconv_out)))
    return GDN_ERR_INVALID;
  const size_t es = esize(cfg->act), eo = out_esize(cfg);
  const size_t HvD = (size_t)cfg->n_v_heads * GDN_HEAD_DIM, nt = (size_t)B * T;
  const size_t C = (size_t)channels(cfg);
  if (overlap(out, nt * HvD * eo, x, nt * C * es) || overlap(out, nt * HvD * eo, z, nt * HvD * es))
    return GDN_ERR_INVALID;
  // the post-conv copy is written while other blocks still read x, z and the pools
  if (postconv_out && (overlap(postconv_out, nt * C * es, x, nt * C * es) ||
                       overlap(postconv_out, nt * C * es, z, nt * HvD * es) ||
                       overlap(postconv_out, nt * C * es, out, nt * HvD * eo)))
    return GDN_ERR_INVALID;
  if (workspace_bytes < 0 || (!workspace && workspace_bytes != 0)) return GDN_ERR_INVALID;
  gdn::StepArgs a = step_args(cfg, B, T);
  a.x = x; a.conv_w = conv_w; a.conv_state = conv_state; a.state = state; a.alpha = alpha;
  a.beta = beta; a.z = z; a.norm_w = norm_w; a.out = out; a.postconv = postconv_out;
  a.slot_idx = slot_idx;
  return from_cuda(gdn::launch_verify(a, (flags & GDN_VERIFY_COMMIT_ALL) != 0, cfg->act,
                                      static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_verify_step_lazy(const gdn_config* cfg, const void* prev_x, const void* prev_alpha,
                                const void* prev_beta, const int32_t* prev_n_keep, int32_t prev_T,
                                const void* x, const void* conv_w, void* conv_state, float* state,
                                const void* alpha, const void* beta, const void* z,
                                const float* norm_w, void* out, const int32_t* slot_idx, int32_t B,
                                int32_t T, void* postconv_out, void* stream) {
  gdn_status st = check_cfg(cfg);
  if (st != GDN_OK) return st;
  if (B < 0 || T < 1 || T > GDN_MAX_DRAFT || prev_T < 1 || prev_T > GDN_MAX_DRAFT)
    return GDN_ERR_INVALID;
  if (B == 0) return GDN_OK;
  if (B > 65535) return GDN_ERR_UNSUPPORTED;
  if (!prev_x || !prev_alpha || !prev_beta || !prev_n_keep || !x || !conv_w || !conv_state ||
      !state || !alpha || !beta || !z || !norm_w || !out || !slot_idx)
    return GDN_ERR_INVALID;
  if (!aligned16(prev_x) || !aligned16(x) || !aligned16(conv_w) || !aligned16(conv_state) ||
      !aligned16(state) || !aligned16(z) || !aligned16(out) || !aligned16(norm_w) ||
      (postconv_out && !aligned16(postconv_out)))
    return GDN_ERR_INVALID;
  const size_t es = esize(cfg->act), eo = out_esize(cfg);
  const size_t HvD = (size_t)cfg->n_v_heads * GDN_HEAD_DIM, C = (size_t)channels(cfg);
  const size_t nt = (size_t)B * T, np = (size_t)B * prev_T;
  if (overlap(out, nt * HvD * eo, x, nt * C * es) || overlap(out, nt * HvD * eo, z, nt * HvD * es) ||
      overlap(out, nt * HvD * eo, prev_x, np * C * es))
    return GDN_ERR_INVALID;
  if (postconv_out && (overlap(postconv_out, nt * C * es, x, nt * C * es) ||
                       overlap(postconv_out, nt * C * es, z, nt * HvD * es) ||
                       overlap(postconv_out, nt * C * es, out, nt * HvD * eo) ||
                       overlap(postconv_out, nt * C * es, prev_x, np * C * es)))
    return GDN_ERR_INVALID;
  gdn::StepArgs a = step_args(cfg, B, T);
  a.x = x; a.conv_w = conv_w; a.conv_state = conv_state; a.state = state; a.alpha = alpha;
  a.beta = beta; a.z = z; a.norm_w = norm_w; a.out = out; a.postconv = postconv_out;
  a.slot_idx = slot_idx; a.n_keep = prev_n_keep;
  a.prev_x = prev_x; a.prev_alpha = prev_alpha; a.prev_beta = prev_beta; a.prev_T = prev_T;
  return from_cuda(gdn::launch_verify_lazy(a, cfg->act, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_commit_layers(const gdn_config* cfg, const gdn_layer_view* layers, int32_t L,
                             const int32_t* slot_idx, const int32_t* n_keep, int32_t B,
                             int32_t T, void* stream) {
  gdn_status st = check_cfg(cfg);
  if (st != GDN_OK) return st;
  if (L < 0 || B < 0 || T < 1 || T > GDN_MAX_DRAFT) return GDN_ERR_INVALID;
  if (L == 0 || B == 0) return GDN_OK;
  if (B > 65535 || L > 65535) return GDN_ERR_UNSUPPORTED;
  if (!layers || !slot_idx || !n_keep || (reinterpret_cast<uintptr_t>(layers) & 7u))
    return GDN_ERR_INVALID;
  gdn::StepArgs a = step_args(cfg, B, T);
  a.q_scale = 1.0f;
  a.slot_idx = slot_idx; a.n_keep = n_keep; a.layers = layers;
  return from_cuda(gdn::launch_commit(a, L, cfg->act, static_cast<cudaStream_t>(stream)));
}

gdn_status gdn_gates(const gdn_config* cfg, const void* a, const void* b, void* alpha,
                     void* beta, int64_t n_tok, void* stream) {
  if (!cfg) return GDN_ERR_INVALID;
  if (cfg->n_v_heads < 1 || n_tok < 0) return GDN_ERR_INVALID;
  if (cfg->gate_dtype != GDN_F32 && cfg->gate_dtype != GDN_BF16) return GDN_ERR_UNSUPPORTED;
  if (n_tok == 0) return GDN_OK;
  if (!a || !b || !alpha || !beta) return GDN_ERR_INVALID;
  const int64_t n = n_tok * cfg->n_v_heads;
  if (n / cfg->n_v_heads != n_tok) return GDN_ERR_INVALID;
  const size_t ge = cfg->gate_dtype == GDN_BF16 ? 2 : 4;
  if ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) | reinterpret_cast<uintptr_t>(alpha) |
       reinterpret_cast<uintptr_t>(beta)) & (ge - 1))
    return GDN_ERR_INVALID;
  const size_t nb = (size_t)n * ge;
  // in place is allowed (alpha = a, beta = b); any other overlap is not
  if ((alpha != a && overlap(alpha, nb, a, nb)) || (beta != b && overlap(beta, nb, b, nb)) ||
      overlap(alpha, nb, beta, nb) || overlap(alpha, nb, b, nb) || overlap(beta, nb, a, nb))
    return GDN_ERR_INVALID;
  return from_cuda(gdn::launch_gates(a, b, alpha, beta, n, cfg->gate_dtype == GDN_BF16,
                                     static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
