// Gated DeltaNet token-mixing path: CPU ORACLE (test infrastructure only).
//
// A plain, slow, single-threaded restatement of what the path computes, used
// by the tests and by the benchmark's CPU-baseline leg to check and time the
// GPU library. It shares no code with the GPU library and is never on the
// product path. One template body serves float and double; the double
// instantiation is the precision reference, the float one evaluates the same
// plain definitions in single precision (each product and each sum rounded
// separately, the library exp) so that its own error can be bounded against
// the double one.
//
// Build: g++ -std=c++17 -O2 -ffp-contract=off -fPIC -shared (no fast-math, no
// FMA contraction: every product and every sum below is rounded separately).
//
// Sources (page title, section):
//   [P1] "perf(gdn): optimize post-conv and causal-conv kernels - #155",
//        maintainer review: the causal conv (width k over c channels, "Blocker"),
//        the 128-lane sum-of-squares tree followed by 1/sqrtf ("Merged ..."),
//        the initial/final conv_state rows of exact chunks ("New issue #305").
//   [P2] same pull request, author's description: exact causal-conv chunk
//        descriptors ("Before starting"), post-conv and conv K4 kernels
//        ("What changed").
//   [P3] "Strata PR #3226": speculative verify over T draft tokens, the
//        output norm after the recurrence, the commit of the accepted prefix of
//        conv_state and recurrent state across layers ("Summary", items 1-3).
//   [DEF] the gated delta rule itself, which the pages name but never write
//        out: S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,
//        o_t = S_t q_t, followed by a z-gated RMSNorm.
//
// Readings where the pages are silent (each is also listed with the design):
//   - head_dim 128, conv width 4, no conv bias; tap 3 multiplies the current
//     token; conv_state holds the 3 previous rows, oldest first.
//   - SiLU follows the conv on every channel; the L2 norm applies to q and k
//     heads only: r = 1/sqrt(sum_sq + eps), eps an argument (1e-6 by default).
//   - v head h reads q/k head h / (Hv/Hk) (contiguous grouping).
//   - the RMSNorm normalises first, then gates: out = o * r * w * silu(z),
//     r = 1/sqrt(mean(o^2) + eps), one weight vector of 128 shared by heads.
//   - o_t uses the updated state; q_scale multiplies o (1.0 reproduces DEF).
//   - a negative slot index marks a padding sequence: nothing is read or
//     written for it.
//   - the gate step (named by [P3] "Root Cause & RED / GREEN Verification",
//     which tests a fused gate kernel against its multi-token form, with no
//     formula) is the workload's own form of the gates: alpha = e^-softplus(a),
//     beta = sigmoid(b), from raw per-(token, v head) projections a, b.
//
// Parity pins (tests/test_oracle_pins.py) fix every function here against
// brute force, closed forms and invariants; see the test file for the list.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

constexpr int D = 128;   // head_dim (dk = dv)
constexpr int KW = 4;    // conv width
constexpr int KS = KW - 1;

// Round to the nearest bfloat16 value (ties to even), computed directly from
// T so that double inputs are not rounded twice.
template <class T> T round_bf16(T v) {
  if (v == T(0) || !std::isfinite(v)) return v;
  const T tiny = std::ldexp(T(1), -126);
  if (std::fabs(v) < tiny) {                       // bf16 subnormal grid 2^-133
    return std::ldexp(std::nearbyint(std::ldexp(v, 133)), -133);
  }
  int e = 0;
  T m = std::frexp(v, &e);                          // v = m * 2^e, 0.5 <= |m| < 1
  T r = std::nearbyint(std::ldexp(m, 8));           // 8 significant bits
  return std::ldexp(r, e - 8);
}

// SiLU, y / (1 + e^-y), with the library exponential, in the oracle's type.
template <class T> T silu(T y) { return y / (T(1) + std::exp(-y)); }

// The canonical sum-of-squares tree over 128 values: 16 groups of 8
// contiguous channels; inside a group the strides 4, 2, 1 are folded, then the
// 16 group sums are folded with strides 8, 4, 2, 1.
template <class T> T tree_sum_sq(const T* v) {
  T g[16];
  for (int grp = 0; grp < 16; ++grp) {
    T e[8];
    for (int j = 0; j < 8; ++j) e[j] = v[8 * grp + j] * v[8 * grp + j];
    T p0 = e[0] + e[4], p1 = e[1] + e[5], p2 = e[2] + e[6], p3 = e[3] + e[7];
    T q0 = p0 + p2, q1 = p1 + p3;
    g[grp] = q0 + q1;
  }
  for (int stride = 8; stride >= 1; stride /= 2)
    for (int i = 0; i < stride; ++i) g[i] = g[i] + g[i + stride];
  return g[0];
}

// [P1 "Merged ..."]: 128-lane sum of squares, then 1/sqrt, then scale.
template <class T> void l2norm_head(T* v, T eps) {
  T ss = tree_sum_sq(v);
  T r = T(1) / std::sqrt(ss + eps);
  for (int i = 0; i < D; ++i) v[i] = v[i] * r;
}

// [P3 output norm] z-gated RMSNorm over one head's 128 outputs.
template <class T> void gated_rmsnorm(const T* o, const T* z, const T* w, T eps, T* out) {
  T ms = tree_sum_sq(o) / T(D);
  T r = T(1) / std::sqrt(ms + eps);
  for (int i = 0; i < D; ++i) out[i] = ((o[i] * r) * w[i]) * silu(z[i]);
}

struct Geo {
  int Hk, Hv, C;
  explicit Geo(int hk, int hv) : Hk(hk), Hv(hv), C((2 * hk + hv) * D) {}
  int q_off(int hk) const { return hk * D; }
  int k_off(int hk) const { return (Hk + hk) * D; }
  int v_off(int h) const { return (2 * Hk + h) * D; }
  int qk_head(int h) const { return h / (Hv / Hk); }
};

// Causal depthwise conv of one channel's padded column xp (3 state rows then
// the tokens): y[t] = sum_j w[j] * xp[t + j], summed from zero in tap order,
// each product and each sum rounded on its own (no fused multiply-add).
template <class T> T conv_tap(const T* w, const T* xp_t) {
  T acc = T(0);
  for (int j = 0; j < KW; ++j) acc = acc + w[j] * xp_t[j];
  return acc;
}

// Post-conv activations of n tokens whose padded columns are given by
// `prev` (3 rows of C, or null for zeros) followed by `x` rows (stride C).
// silu/l2: apply the activation / the q,k L2 norm.  Output y rows (stride C).
template <class T>
void conv_block(const Geo& g, const T* x, int64_t n, const T* w, const T* prev,
                int silu_on, int l2_on, T eps, T* y) {
  std::vector<T> xp(n + KS);
  for (int c = 0; c < g.C; ++c) {
    for (int r = 0; r < KS; ++r) xp[r] = prev ? prev[(int64_t)r * g.C + c] : T(0);
    for (int64_t t = 0; t < n; ++t) xp[KS + t] = x[t * g.C + c];
    for (int64_t t = 0; t < n; ++t) {
      T a = conv_tap(w + (int64_t)c * KW, &xp[t]);
      y[t * g.C + c] = silu_on ? silu(a) : a;
    }
  }
  if (l2_on) {
    for (int64_t t = 0; t < n; ++t)
      for (int h = 0; h < 2 * g.Hk; ++h) l2norm_head(y + t * g.C + (int64_t)h * D, eps);
  }
}

// The last 3 rows of (prev ++ x[0:n]) for every channel: the committed
// conv_state. prev null means zero rows.
template <class T>
void conv_tail(const Geo& g, const T* prev, const T* x, int64_t n, T* out) {
  for (int r = 0; r < KS; ++r) {
    int64_t idx = n + r;                 // index into (prev ++ x)
    for (int c = 0; c < g.C; ++c) {
      T v;
      if (idx >= KS) v = x[(idx - KS) * g.C + c];
      else v = prev ? prev[(int64_t)idx * g.C + c] : T(0);
      out[(int64_t)r * g.C + c] = v;
    }
  }
}

// [DEF] one token of the gated delta rule on one head, in the expanded form
// u = S k;  S <- a S + b (v - a u) k^T  (= a S (I - b k k^T) + b v k^T);
// o = q_scale * S q with the updated S.
template <class T>
void delta_token(T* S, const T* q, const T* k, const T* v, T a, T b, T q_scale, T* o) {
  for (int i = 0; i < D; ++i) {
    T* row = S + (int64_t)i * D;
    T u = T(0);
    for (int j = 0; j < D; ++j) u = u + row[j] * k[j];
    T d = b * (v[i] - a * u);
    for (int j = 0; j < D; ++j) row[j] = a * row[j] + d * k[j];
  }
  for (int i = 0; i < D; ++i) {
    const T* row = S + (int64_t)i * D;
    T acc = T(0);
    for (int j = 0; j < D; ++j) acc = acc + row[j] * q[j];
    o[i] = q_scale * acc;
  }
}

// Token-by-token recurrence over n tokens of one sequence (all v heads).
// qkv rows stride C; alpha/beta rows stride Hv; z/out rows stride Hv*D.
template <class T>
void recurrence_seq(const Geo& g, const T* qkv, const T* alpha, const T* beta, const T* z,
                    const T* norm_w, T* S /* [Hv][D][D] */, int64_t n, T q_scale, T eps,
                    T* out, T* o_raw) {
  std::vector<T> o(D);
  const int64_t HvD = (int64_t)g.Hv * D;
  for (int64_t t = 0; t < n; ++t) {
    const T* row = qkv + t * g.C;
    for (int h = 0; h < g.Hv; ++h) {
      int hk = g.qk_head(h);
      delta_token(S + (int64_t)h * D * D, row + g.q_off(hk), row + g.k_off(hk), row + g.v_off(h),
                  alpha[t * g.Hv + h], beta[t * g.Hv + h], q_scale, o.data());
      if (o_raw) std::memcpy(o_raw + t * HvD + (int64_t)h * D, o.data(), sizeof(T) * D);
      if (out) gated_rmsnorm(o.data(), z + t * HvD + (int64_t)h * D, norm_w, eps,
                             out + t * HvD + (int64_t)h * D);
    }
  }
}

// The chunked (WY) form of the same recurrence over one sequence, a second,
// independent restatement used to check the first and the GPU's chunked path.
// Inside a chunk, with g_t = sum_{s<=t} log a_s (chunk-local):
//   A_ts = b_t exp(g_t - g_s) (k_t . k_s), s < t
//   d_t  = b_t v_t - b_t exp(g_t) S0 k_t - sum_{s<t} A_ts d_s
//   o_t  = exp(g_t) S0 q_t + sum_{s<=t} exp(g_t - g_s) (k_s . q_t) d_s
//   S    = exp(g_last) S0 + sum_s exp(g_last - g_s) d_s k_s^T
template <class T>
void chunked_seq(const Geo& g, const T* qkv, const T* alpha, const T* beta, const T* z,
                 const T* norm_w, T* Sall, int64_t n, int chunk, T q_scale, T eps,
                 T* out, T* o_raw) {
  const int64_t HvD = (int64_t)g.Hv * D;
  std::vector<T> G(chunk), A((size_t)chunk * chunk), Dm((size_t)chunk * D), o(D), S0k(D), S0q(D);
  for (int h = 0; h < g.Hv; ++h) {
    T* S = Sall + (int64_t)h * D * D;
    const int hk = g.qk_head(h);
    for (int64_t c0 = 0; c0 < n; c0 += chunk) {
      const int m = (int)std::min<int64_t>(chunk, n - c0);
      auto qv = [&](int t) { return qkv + (c0 + t) * g.C + g.q_off(hk); };
      auto kv = [&](int t) { return qkv + (c0 + t) * g.C + g.k_off(hk); };
      auto vv = [&](int t) { return qkv + (c0 + t) * g.C + g.v_off(h); };
      auto dot = [](const T* a, const T* b) { T s = T(0); for (int j = 0; j < D; ++j) s = s + a[j] * b[j]; return s; };
      T acc = T(0);
      for (int t = 0; t < m; ++t) { acc = acc + std::log(alpha[(c0 + t) * g.Hv + h]); G[t] = acc; }
      for (int t = 0; t < m; ++t)
        for (int s = 0; s < t; ++s)
          A[(size_t)t * chunk + s] = beta[(c0 + t) * g.Hv + h] * std::exp(G[t] - G[s]) * dot(kv(t), kv(s));
      // forward substitution for the deltas d_t (rows of Dm)
      for (int t = 0; t < m; ++t) {
        const T b = beta[(c0 + t) * g.Hv + h];
        const T gt = std::exp(G[t]);
        for (int i = 0; i < D; ++i) S0k[i] = dot(S + (int64_t)i * D, kv(t));
        for (int i = 0; i < D; ++i) {
          T r = b * vv(t)[i] - b * gt * S0k[i];
          for (int s = 0; s < t; ++s) r = r - A[(size_t)t * chunk + s] * Dm[(size_t)s * D + i];
          Dm[(size_t)t * D + i] = r;
        }
      }
      // outputs
      for (int t = 0; t < m; ++t) {
        const T gt = std::exp(G[t]);
        for (int i = 0; i < D; ++i) S0q[i] = dot(S + (int64_t)i * D, qv(t));
        for (int i = 0; i < D; ++i) {
          T acc2 = gt * S0q[i];
          for (int s = 0; s <= t; ++s)
            acc2 = acc2 + std::exp(G[t] - G[s]) * dot(kv(s), qv(t)) * Dm[(size_t)s * D + i];
          o[i] = q_scale * acc2;
        }
        const int64_t tt = c0 + t;
        if (o_raw) std::memcpy(o_raw + tt * HvD + (int64_t)h * D, o.data(), sizeof(T) * D);
        if (out) gated_rmsnorm(o.data(), z + tt * HvD + (int64_t)h * D, norm_w, eps,
                               out + tt * HvD + (int64_t)h * D);
      }
      // state at the end of the chunk
      const T gl = std::exp(G[m - 1]);
      for (int i = 0; i < D; ++i)
        for (int j = 0; j < D; ++j) {
          T acc3 = gl * S[(int64_t)i * D + j];
          for (int s = 0; s < m; ++s)
            acc3 = acc3 + std::exp(G[m - 1] - G[s]) * Dm[(size_t)s * D + i] * kv(s)[j];
          S[(int64_t)i * D + j] = acc3;
        }
    }
  }
}

// The gate step: alpha = exp(-softplus(a)), softplus(a) = log(1 + e^a), and
// beta = 1 / (1 + e^-b), for n elements. softplus is taken as a + log(1 + e^-a)
// for a > 0 so that e^a is never formed for large a (the same value in exact
// arithmetic); log1p keeps the small-argument digits.
template <class T> void gates(const T* a, const T* b, int64_t n, T* alpha, T* beta) {
  for (int64_t i = 0; i < n; ++i) {
    const T x = a[i];
    const T sp = x > T(0) ? x + std::log1p(std::exp(-x)) : std::log1p(std::exp(x));
    alpha[i] = std::exp(-sp);
    beta[i] = T(1) / (T(1) + std::exp(-b[i]));
  }
}

}  // namespace

// ============================================================== C entry points
// Every function below exists as name_f32 (T = float) and name_f64 (T = double).
// Arrays are dense row-major in the layouts of the GPU library; activation
// arrays are passed already widened to T.

#define ORACLE_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

// [P1 "Blocker", "New issue #305"; P2 "Before starting"] varlen causal conv.
// For every sequence s with slot_idx[s] >= 0: the padded column is
// (conv_state[slot] if has_init[s] else zeros) ++ x rows of s; y rows of s get
// the activations; conv_state[slot] receives the last 3 padded rows, written
// after every read of the sequence.
template <class T>
void conv_fwd(const T* x, int64_t n_tok, int Hk, int Hv, const T* w, T* conv_state,
              const int32_t* slot_idx, const int32_t* cu, const uint8_t* has_init, int n_seq,
              int silu_on, int l2_on, T eps, T* y) {
  (void)n_tok;
  Geo g(Hk, Hv);
  std::vector<T> tail((size_t)KS * g.C);
  for (int s = 0; s < n_seq; ++s) {
    const int slot = slot_idx[s];
    if (slot < 0) continue;
    const int64_t t0 = cu[s], n = cu[s + 1] - cu[s];
    T* st = conv_state + (int64_t)slot * KS * g.C;
    const T* prev = has_init[s] ? st : nullptr;
    conv_block(g, x + t0 * g.C, n, w, prev, silu_on, l2_on, eps, y + t0 * g.C);
    conv_tail(g, prev, x + t0 * g.C, n, tail.data());
    std::memcpy(st, tail.data(), sizeof(T) * tail.size());
  }
}

// [DEF] token-by-token (chunk == 0) or chunked (chunk >= 1) prefill of the
// recurrence over varlen sequences; state[slot] is read when has_init[s] and
// always receives the final state.
template <class T>
void prefill(const T* qkv, const T* alpha, const T* beta, const T* z, const T* norm_w,
             T* state, const int32_t* slot_idx, const int32_t* cu, const uint8_t* has_init,
             int n_seq, int Hk, int Hv, T q_scale, T eps, int chunk, T* out, T* o_raw) {
  Geo g(Hk, Hv);
  const int64_t HvD = (int64_t)Hv * D, SS = (int64_t)Hv * D * D;
  std::vector<T> S(SS);
  for (int s = 0; s < n_seq; ++s) {
    const int slot = slot_idx[s];
    if (slot < 0) continue;
    const int64_t t0 = cu[s], n = cu[s + 1] - cu[s];
    if (has_init[s]) std::memcpy(S.data(), state + slot * SS, sizeof(T) * SS);
    else std::fill(S.begin(), S.end(), T(0));
    T* outp = out ? out + t0 * HvD : nullptr;
    T* orp = o_raw ? o_raw + t0 * HvD : nullptr;
    if (chunk <= 0)
      recurrence_seq(g, qkv + t0 * g.C, alpha + t0 * Hv, beta + t0 * Hv, z + t0 * HvD, norm_w,
                     S.data(), n, q_scale, eps, outp, orp);
    else
      chunked_seq(g, qkv + t0 * g.C, alpha + t0 * Hv, beta + t0 * Hv, z + t0 * HvD, norm_w,
                  S.data(), n, chunk, q_scale, eps, outp, orp);
    std::memcpy(state + slot * SS, S.data(), sizeof(T) * SS);
  }
}

// Post-conv activations of T draft tokens of batch entry b from its
// conv_state; rounded to the activation type when round_act (the reading of
// the verify / commit phases is that the fused kernels feed the recurrence
// unrounded values, so the tests pass round_act = 0; 1 models activations
// that went through memory, as the prefill's do).
template <class T>
void draft_activations(const Geo& g, const T* xb, int Tn, const T* w, const T* st, T eps,
                       int round_act, T* qkv) {
  const int64_t n = (int64_t)Tn * g.C;
  conv_block(g, xb, Tn, w, st, 1, 1, eps, qkv);
  if (round_act)
    for (int64_t i = 0; i < n; ++i) qkv[i] = round_bf16(qkv[i]);
}

// [P3 "Summary"; DEF] speculative verify of T draft tokens per batch entry:
// outputs of every draft token from the current conv_state and state, which
// are left untouched unless commit_all (then both advance by all T tokens).
template <class T>
void verify(const T* x, const T* w, T* conv_state, T* state, const T* alpha, const T* beta,
            const T* z, const T* norm_w, const int32_t* slot_idx, int B, int Tn, int Hk, int Hv,
            T q_scale, T eps, int round_act, int commit_all, T* out, T* postconv, T* o_raw) {
  Geo g(Hk, Hv);
  const int64_t HvD = (int64_t)Hv * D, SS = (int64_t)Hv * D * D;
  std::vector<T> qkv((size_t)Tn * g.C), S(SS), tail((size_t)KS * g.C);
  for (int b = 0; b < B; ++b) {
    const int slot = slot_idx[b];
    if (slot < 0) continue;
    const T* xb = x + (int64_t)b * Tn * g.C;
    T* st = conv_state + (int64_t)slot * KS * g.C;
    draft_activations(g, xb, Tn, w, st, eps, round_act, qkv.data());
    if (postconv) std::memcpy(postconv + (int64_t)b * Tn * g.C, qkv.data(), sizeof(T) * qkv.size());
    std::memcpy(S.data(), state + slot * SS, sizeof(T) * SS);
    recurrence_seq(g, qkv.data(), alpha + (int64_t)b * Tn * Hv, beta + (int64_t)b * Tn * Hv,
                   z + (int64_t)b * Tn * HvD, norm_w, S.data(), Tn, q_scale, eps,
                   out + (int64_t)b * Tn * HvD, o_raw ? o_raw + (int64_t)b * Tn * HvD : nullptr);
    if (commit_all) {
      std::memcpy(state + slot * SS, S.data(), sizeof(T) * SS);
      conv_tail(g, st, xb, Tn, tail.data());
      std::memcpy(st, tail.data(), sizeof(T) * tail.size());
    }
  }
}

// [P3 "Summary" item 1] commit of the accepted prefix of one layer: for each
// batch entry with 0 <= n_keep[b] <= T, conv_state <- last 3 rows of
// (conv_state ++ x[b, 0:n]) and state <- the state after those n tokens.
// n_keep == 0 leaves both untouched; entries with n_keep outside [0, T] are
// skipped.
template <class T>
void commit(const T* x, const T* alpha, const T* beta, const T* w, T* conv_state, T* state,
            const int32_t* slot_idx, const int32_t* n_keep, int B, int Tn, int Hk, int Hv,
            T eps, int round_act) {
  Geo g(Hk, Hv);
  const int64_t SS = (int64_t)Hv * D * D;
  std::vector<T> qkv((size_t)Tn * g.C), S(SS), tail((size_t)KS * g.C);
  for (int b = 0; b < B; ++b) {
    const int slot = slot_idx[b];
    const int n = n_keep[b];
    if (slot < 0 || n <= 0 || n > Tn) continue;
    const T* xb = x + (int64_t)b * Tn * g.C;
    T* st = conv_state + (int64_t)slot * KS * g.C;
    draft_activations(g, xb, n, w, st, eps, round_act, qkv.data());
    std::memcpy(S.data(), state + slot * SS, sizeof(T) * SS);
    recurrence_seq<T>(g, qkv.data(), alpha + (int64_t)b * Tn * Hv, beta + (int64_t)b * Tn * Hv,
                      nullptr, nullptr, S.data(), n, T(1), eps, nullptr, nullptr);
    std::memcpy(state + slot * SS, S.data(), sizeof(T) * SS);
    conv_tail(g, st, xb, n, tail.data());
    std::memcpy(st, tail.data(), sizeof(T) * tail.size());
  }
}

}  // namespace

#define ORACLE_INSTANTIATE(T, SUF)                                                              \
  ORACLE_EXPORT void oracle_conv_fwd_##SUF(const T* x, int64_t n_tok, int Hk, int Hv,          \
      const T* w, T* conv_state, const int32_t* slot_idx, const int32_t* cu,                    \
      const uint8_t* has_init, int n_seq, int silu_on, int l2_on, T eps, T* y) {                \
    conv_fwd<T>(x, n_tok, Hk, Hv, w, conv_state, slot_idx, cu, has_init, n_seq, silu_on, l2_on, \
                eps, y);                                                                        \
  }                                                                                             \
  ORACLE_EXPORT void oracle_l2norm_##SUF(T* y, int64_t n_tok, int Hk, int Hv, T eps) {          \
    Geo g(Hk, Hv);                                                                              \
    for (int64_t t = 0; t < n_tok; ++t)                                                         \
      for (int h = 0; h < 2 * Hk; ++h) l2norm_head(y + t * g.C + (int64_t)h * D, eps);          \
  }                                                                                             \
  ORACLE_EXPORT T oracle_tree_sum_sq_##SUF(const T* v) { return tree_sum_sq(v); }               \
  ORACLE_EXPORT void oracle_gated_rmsnorm_##SUF(const T* o, const T* z, const T* w, T eps,      \
                                                T* out) {                                       \
    gated_rmsnorm(o, z, w, eps, out);                                                           \
  }                                                                                             \
  ORACLE_EXPORT void oracle_silu_##SUF(T* v, int64_t n) {                                       \
    for (int64_t i = 0; i < n; ++i) v[i] = silu(v[i]);                                          \
  }                                                                                             \
  ORACLE_EXPORT void oracle_round_bf16_##SUF(T* v, int64_t n) {                                 \
    for (int64_t i = 0; i < n; ++i) v[i] = round_bf16(v[i]);                                    \
  }                                                                                             \
  ORACLE_EXPORT void oracle_prefill_##SUF(const T* qkv, const T* alpha, const T* beta,         \
      const T* z, const T* norm_w, T* state, const int32_t* slot_idx, const int32_t* cu,        \
      const uint8_t* has_init, int n_seq, int Hk, int Hv, T q_scale, T eps, int chunk, T* out,  \
      T* o_raw) {                                                                               \
    prefill<T>(qkv, alpha, beta, z, norm_w, state, slot_idx, cu, has_init, n_seq, Hk, Hv,       \
               q_scale, eps, chunk, out, o_raw);                                                \
  }                                                                                             \
  ORACLE_EXPORT void oracle_verify_##SUF(const T* x, const T* w, T* conv_state, T* state,      \
      const T* alpha, const T* beta, const T* z, const T* norm_w, const int32_t* slot_idx,      \
      int B, int Tn, int Hk, int Hv, T q_scale, T eps, int round_act, int commit_all, T* out,   \
      T* postconv, T* o_raw) {                                                                  \
    verify<T>(x, w, conv_state, state, alpha, beta, z, norm_w, slot_idx, B, Tn, Hk, Hv,         \
              q_scale, eps, round_act, commit_all, out, postconv, o_raw);                       \
  }                                                                                             \
  ORACLE_EXPORT void oracle_gates_##SUF(const T* a, const T* b, int64_t n, T* alpha, T* beta) { \
    gates<T>(a, b, n, alpha, beta);                                                             \
  }                                                                                             \
  ORACLE_EXPORT void oracle_commit_##SUF(const T* x, const T* alpha, const T* beta,            \
      const T* w, T* conv_state, T* state, const int32_t* slot_idx, const int32_t* n_keep,      \
      int B, int Tn, int Hk, int Hv, T eps, int round_act) {                                    \
    commit<T>(x, alpha, beta, w, conv_state, state, slot_idx, n_keep, B, Tn, Hk, Hv, eps,       \
              round_act);                                                                       \
  }

ORACLE_INSTANTIATE(float, f32)
ORACLE_INSTANTIATE(double, f64)
