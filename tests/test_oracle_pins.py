"""Pins of the CPU oracle against brute force, closed forms and invariants.

Each test fixes one part of the oracle to something other than itself, so
that a plausible slip (a dropped term, a wrong sign or index, a transposed
operand, a changed reduction order) fails at least one of them:

  P1  conv = exact 4-term sums (rational arithmetic) within 7 roundings;
      has_init=0 = zero-padded np.convolve; SiLU = y / (1 + e^-y), the float
      instantiation within 4 ulp of the double one
  P2  delta conv weights: pass-through of the current token and a 3-row shift
      that reads the conv_state (pins tap orientation and state row order)
  P3  L2 norm: unit norm, tree sum within the pairwise bound of the exact sum,
      exact order-revealing inputs, and the sequential fold it must not be
  P4  beta = 0: S_t = (prod alpha) S_0 and o_t = S_t q_t
  P5  beta = 1 with unit keys: the delta rule writes v exactly (S_t k_t = v_t)
  P6  one-hot keys, alpha = 1, beta = 1/2: bitwise column update
  P7  chunked WY form = token-by-token form for chunks 1, 2, 7, 64
  P8  phases: split prefill, prefill + verify, commit of an accepted prefix
  P9  gated RMSNorm closed forms
  P10 float instantiation against double
  DEF the matrix form of the gated delta rule
  BF  bfloat16 rounding against torch's conversion
  GT  the gate step: alpha = exp(-softplus(a)) equals the logistic function of -a
      (scipy's expit), beta = expit(b), closed values at 0, saturation without
      overflow, the float instantiation against double
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from gated_deltanet_linear_12_gb300 import synthetic as syn

D = 128


def _tiny_prefill(lens=(5, 2, 9), Hk=1, Hv=2, seed=7, init=(1, 0, 1), gate="uniform"):
    return syn.prefill_inputs(list(lens), Hk, Hv, "f32", seed=seed, init_mask=np.array(init),
                              gate_form=gate)


# ------------------------------------------------------------------ P1
def test_p1_conv_explicit_sums(orc):
    inp = _tiny_prefill()
    x, w, cs = inp["x"].astype(np.float64), inp["conv_w"].astype(np.float64), inp["conv_state"]
    y, st = orc.conv_fwd(inp["x"], inp["conv_w"], cs, inp["slot_idx"], inp["cu_seqlens"],
                         inp["has_init_conv"], inp["Hk"], inp["Hv"], silu=False, l2norm=False)
    cu = inp["cu_seqlens"]
    for s in range(inp["n_seq"]):
        slot = inp["slot_idx"][s]
        t0, n = cu[s], cu[s + 1] - cu[s]
        prev = cs[slot].astype(np.float64) if inp["has_init_conv"][s] else np.zeros((3, inp["C"]))
        for c in range(0, inp["C"], 37):
            col = [prev[0, c], prev[1, c], prev[2, c]] + [x[t0 + t, c] for t in range(n)]
            for t in range(n):
                terms = [Fraction(float(w[c, j])) * Fraction(float(col[t + j])) for j in range(4)]
                exact = sum(terms)
                # four rounded products and three rounded sums: 7 roundings
                bound = 7 * 2.0 ** -53 * float(sum(abs(v) for v in terms))
                assert abs(Fraction(float(y[t0 + t, c])) - exact) <= Fraction(bound)
            # committed state = last three rows of the padded column
            assert [st[slot, r, c] for r in range(3)] == col[n:n + 3]


def test_p1_conv_zero_init_is_zero_padded_convolution(orc):
    inp = _tiny_prefill(lens=(11,), init=(0,))
    y, _ = orc.conv_fwd(inp["x"], inp["conv_w"], inp["conv_state"], inp["slot_idx"],
                        inp["cu_seqlens"], inp["has_init_conv"], inp["Hk"], inp["Hv"],
                        silu=False, l2norm=False)
    x = inp["x"].astype(np.float64)
    w = inp["conv_w"].astype(np.float64)
    for c in range(inp["C"]):
        # y[t] = sum_j w[j] x[t - 3 + j]  ==  (x * reversed(w))[t]
        full = np.convolve(x[:, c], w[c, ::-1])[: x.shape[0]]
        np.testing.assert_allclose(y[:, c], full, rtol=1e-12, atol=1e-12)


def test_p1_silu_applied_after_conv(orc):
    inp = _tiny_prefill(lens=(4,), init=(1,))
    args = (inp["x"], inp["conv_w"], inp["conv_state"], inp["slot_idx"], inp["cu_seqlens"],
            inp["has_init_conv"], inp["Hk"], inp["Hv"])
    pre, _ = orc.conv_fwd(*args, silu=False, l2norm=False)
    post, _ = orc.conv_fwd(*args, silu=True, l2norm=False)
    want = np.vectorize(lambda a: a / (1.0 + math.exp(-a)))(pre)
    np.testing.assert_allclose(post, want, rtol=1e-15, atol=0)


def test_p1_f32_silu_within_four_ulp(orc):
    """The float instantiation's SiLU (library expf, a rounded add and divide)
    against y / (1 + math.exp(-y)) in double."""
    ys = np.concatenate([np.linspace(-87.0, 88.0, 400001, dtype=np.float32),
                         np.float32([0.0, -0.0, 1e-8, -1e-8, 0.34657359, -0.34657359, 1e-30])])
    got = orc.silu(ys, prec="f32").astype(np.float64)
    for y, g in zip(ys[::37].astype(np.float64), got[::37]):
        want = y / (1.0 + math.exp(-y))
        ulp = float(np.spacing(np.float32(abs(want))))
        assert abs(g - want) <= 4 * ulp, (y, g, want)


# ------------------------------------------------------------------ P2
@pytest.mark.parametrize("prec", ["f64", "f32"])
def test_p2_delta_weights(orc, prec):
    inp = _tiny_prefill(lens=(6, 2), init=(1, 1))
    C = inp["C"]
    x = inp["x"]
    cs = inp["conv_state"]
    cu = inp["cu_seqlens"]
    common = (cs, inp["slot_idx"], cu, inp["has_init_conv"], inp["Hk"], inp["Hv"])
    w_id = np.zeros((C, 4), np.float32)
    w_id[:, 3] = 1.0
    y, _ = orc.conv_fwd(x, w_id, *common, silu=False, l2norm=False, prec=prec)
    assert np.array_equal(y, x.astype(y.dtype))
    w_sh = np.zeros((C, 4), np.float32)
    w_sh[:, 0] = 1.0
    y, st = orc.conv_fwd(x, w_sh, *common, silu=False, l2norm=False, prec=prec)
    for s in range(2):
        slot = inp["slot_idx"][s]
        padded = np.concatenate([cs[slot], x[cu[s]:cu[s + 1]]], axis=0)
        n = cu[s + 1] - cu[s]
        assert np.array_equal(y[cu[s]:cu[s + 1]], padded[:n].astype(y.dtype))
        assert np.array_equal(st[slot], padded[n:n + 3].astype(y.dtype))


def test_p2_padding_sequence_untouched(orc):
    inp = _tiny_prefill(lens=(3, 4), init=(1, 1))
    slots = inp["slot_idx"].copy()
    slots[1] = -1
    y, st = orc.conv_fwd(inp["x"], inp["conv_w"], inp["conv_state"], slots, inp["cu_seqlens"],
                         inp["has_init_conv"], inp["Hk"], inp["Hv"])
    assert np.all(y[3:] == 0)
    untouched = [i for i in range(st.shape[0]) if i != slots[0]]
    assert np.array_equal(st[untouched], inp["conv_state"][untouched].astype(np.float64))


# ------------------------------------------------------------------ P3
def test_p3_unit_norm_and_v_untouched(orc):
    rows = syn.random_f32_rows(64, syn.channels(2, 3), seed=11)
    out = orc.l2norm(rows, 2, 3, prec="f32")
    for h in range(4):
        n = np.linalg.norm(out[:, h * D:(h + 1) * D].astype(np.float64), axis=1)
        assert np.all(np.abs(n - 1.0) < 2.0 ** -20)
    assert np.array_equal(out[:, 4 * D:], rows[:, 4 * D:])


@pytest.mark.parametrize("c", [1e-4, -2e-4, 0.5])
def test_p3_constant_vector_closed_form(orc, c):
    """q = c*1: ss = 128 c^2, so q_hat = c / sqrt(128 c^2 + eps) (eps inside the root)."""
    eps = 1e-6
    rows = np.zeros((1, syn.channels(1, 1)))
    rows[0, :2 * D] = c
    out = orc.l2norm(rows, 1, 1, eps=eps)
    np.testing.assert_allclose(out[0, :2 * D], c / math.sqrt(128 * c * c + eps), rtol=1e-14)


def test_p3_tree_within_pairwise_bound(orc):
    rows = syn.random_f32_rows(200, D, seed=12, scale=3.0)
    u = 2.0 ** -24
    for r in rows:
        exact = math.fsum(float(a) * float(a) for a in r)
        got = float(orc.tree_sum_sq(r, prec="f32"))
        # 128 terms summed by a depth-7 tree, plus the rounding of each square
        assert abs(got - exact) <= 8 * u * exact * (1 + 8 * u)


def _order_probe(ones_at):
    v = np.zeros(D, np.float32)
    v[0] = 2.0 ** 12                      # square 2^24: spacing 2 above it in f32
    for i in ones_at:
        v[i] = 1.0
    return v


@pytest.mark.parametrize("ones_at,expect", [
    # a single 1 meeting 2^24 is absorbed (tie to even)
    ((4,), 2.0 ** 24),
    ((1,), 2.0 ** 24),
    # 1s at channels 1 and 5 meet each other first (stride 4), then as 2
    ((1, 5), 2.0 ** 24 + 2),
    # channels 4 and 2: 4 meets channel 0 first, 2 meets 6 (zero), so both vanish
    ((4, 2), 2.0 ** 24),
    # groups 1 and 9 meet at stride 8 before reaching group 0
    ((8, 72), 2.0 ** 24 + 2),
    # groups 1 and 2 reach group 0 separately: both absorbed
    ((8, 16), 2.0 ** 24),
    # groups 2 and 3 meet at stride 1 only after group 2 met group 0
    ((16, 24), 2.0 ** 24),
    # groups 1 and 3 meet at stride 2, then join group 0 as 2
    ((8, 24), 2.0 ** 24 + 2),
])
def test_p3_tree_order_exact(orc, ones_at, expect):
    assert float(orc.tree_sum_sq(_order_probe(ones_at), prec="f32")) == expect


def test_p3_sequential_fold_is_a_different_order(orc):
    """The rejected sequential fold changes the f32 result in many rows."""
    rows = syn.random_f32_rows(20000, D, seed=13)
    diff = 0
    for r in rows[:4000]:
        seq = np.float32(0)
        for a in r:
            seq = np.float32(seq + np.float32(a * a))
        if seq != np.float32(orc.tree_sum_sq(r, prec="f32")):
            diff += 1
    assert diff > 0


# ------------------------------------------------------------------ helpers
def _raw_qkv(n, Hk, Hv, seed, unit_k=True):
    """Random post-conv rows with unit-norm q and k heads (numpy only)."""
    rng = np.random.default_rng(seed)
    C = syn.channels(Hk, Hv)
    q = rng.standard_normal((n, C))
    if unit_k:
        for h in range(2 * Hk):
            blk = q[:, h * D:(h + 1) * D]
            q[:, h * D:(h + 1) * D] = blk / np.linalg.norm(blk, axis=1, keepdims=True)
    return q


def _run_prefill(orc, qkv, alpha, beta, S0, Hk, Hv, chunk=0, prec="f64", z=None, w=None):
    n = qkv.shape[0]
    z = np.zeros((n, Hv * D)) if z is None else z
    w = np.ones(D) if w is None else w
    st = S0[None].copy()
    return orc.prefill(qkv, alpha, beta, z, w, st, [0], [0, n], [1], Hk, Hv, chunk=chunk,
                       prec=prec, want_raw=True)


# ------------------------------------------------------------------ P4
def test_p4_beta_zero_is_pure_decay(orc):
    Hk, Hv, n = 1, 2, 9
    rng = np.random.default_rng(21)
    qkv = _raw_qkv(n, Hk, Hv, 22)
    alpha = rng.uniform(0.5, 1.0, (n, Hv))
    beta = np.zeros((n, Hv))
    S0 = rng.standard_normal((Hv, D, D))
    _, S, raw = _run_prefill(orc, qkv, alpha, beta, S0, Hk, Hv)
    np.testing.assert_allclose(S[0], S0 * np.prod(alpha, axis=0)[:, None, None], rtol=1e-13)
    for t in range(n):
        for h in range(Hv):
            St = S0[h] * np.prod(alpha[:t + 1, h])
            np.testing.assert_allclose(raw[t, h * D:(h + 1) * D], St @ qkv[t, :D], rtol=1e-12,
                                       atol=1e-12)


# ------------------------------------------------------------------ P5
def test_p5_delta_rule_writes_exactly(orc):
    Hk, Hv, n = 1, 2, 12
    rng = np.random.default_rng(31)
    qkv = _raw_qkv(n, Hk, Hv, 32)
    qkv[:, :D] = qkv[:, D:2 * D]           # q_t = k_t so o_t = S_t k_t
    alpha = rng.uniform(0.1, 1.0, (n, Hv))
    beta = np.ones((n, Hv))
    S0 = rng.standard_normal((Hv, D, D))
    _, _, raw = _run_prefill(orc, qkv, alpha, beta, S0, Hk, Hv)
    for h in range(Hv):
        np.testing.assert_allclose(raw[:, h * D:(h + 1) * D], qkv[:, (2 + h) * D:(3 + h) * D],
                                   rtol=1e-11, atol=1e-11)


# ------------------------------------------------------------------ P6
@pytest.mark.parametrize("prec", ["f64", "f32"])
def test_p6_one_hot_keys_bitwise(orc, prec):
    Hk, Hv, n = 1, 1, 6
    T = np.float64 if prec == "f64" else np.float32
    rng = np.random.default_rng(41)
    C = syn.channels(Hk, Hv)
    qkv = np.zeros((n, C), T)
    cols = [3, 77, 3, 127, 0, 77]
    for t, j in enumerate(cols):
        qkv[t, D + j] = 1.0
        qkv[t, :D] = rng.standard_normal(D)
        qkv[t, 2 * D:] = rng.standard_normal(D)
    alpha = np.ones((n, Hv), T)
    beta = np.full((n, Hv), 0.5, T)
    S0 = rng.standard_normal((1, D, D)).astype(T)
    _, S, _ = _run_prefill(orc, qkv, alpha, beta, S0, Hk, Hv, prec=prec)
    want = S0[0].copy()
    half = T(0.5)
    for t, j in enumerate(cols):
        v = qkv[t, 2 * D:]
        want[:, j] = want[:, j] + half * (v - want[:, j])
    assert np.array_equal(S[0, 0], want)


# ------------------------------------------------------------------ DEF
def test_definition_matrix_form(orc):
    Hk, Hv, n = 1, 2, 7
    rng = np.random.default_rng(51)
    qkv = _raw_qkv(n, Hk, Hv, 52)
    alpha = rng.uniform(0.3, 1.0, (n, Hv))
    beta = rng.uniform(0.0, 1.0, (n, Hv))
    S0 = rng.standard_normal((Hv, D, D))
    _, S, raw = _run_prefill(orc, qkv, alpha, beta, S0, Hk, Hv)
    I = np.eye(D)
    for h in range(Hv):
        St = S0[h].copy()
        for t in range(n):
            q, k, v = qkv[t, :D], qkv[t, D:2 * D], qkv[t, (2 + h) * D:(3 + h) * D]
            St = alpha[t, h] * St @ (I - beta[t, h] * np.outer(k, k)) + beta[t, h] * np.outer(v, k)
            np.testing.assert_allclose(raw[t, h * D:(h + 1) * D], St @ q, rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(S[0, h], St, rtol=1e-10, atol=1e-10)


def test_grouping_two_v_heads_share_one_qk_head(orc):
    """v heads 0,1 read q/k head 0 and v heads 2,3 read head 1 (Hv/Hk = 2)."""
    Hk, Hv, n = 2, 4, 3
    rng = np.random.default_rng(55)
    qkv = _raw_qkv(n, Hk, Hv, 56)
    alpha = rng.uniform(0.5, 1.0, (n, Hv))
    beta = rng.uniform(0.0, 1.0, (n, Hv))
    S0 = rng.standard_normal((Hv, D, D))
    _, S, _ = _run_prefill(orc, qkv, alpha, beta, S0, Hk, Hv)
    for h in range(Hv):
        hk = h // 2
        sub = np.concatenate([qkv[:, hk * D:(hk + 1) * D], qkv[:, (Hk + hk) * D:(Hk + hk + 1) * D],
                              qkv[:, (2 * Hk + h) * D:(2 * Hk + h + 1) * D]], axis=1)
        _, S1, _ = _run_prefill(orc, sub, alpha[:, h:h + 1], beta[:, h:h + 1], S0[h:h + 1], 1, 1)
        assert np.array_equal(S1[0, 0], S[0, h])


# ------------------------------------------------------------------ P7
@pytest.mark.parametrize("chunk", [1, 2, 7, 64])
def test_p7_chunked_equals_token_form(orc, chunk):
    inp = syn.prefill_inputs([5, 70, 1], 1, 2, "f32", seed=61, init_mask=np.array([1, 0, 1]),
                             gate_form="softplus")
    y, _ = orc.conv_fwd(inp["x"], inp["conv_w"], inp["conv_state"], inp["slot_idx"],
                        inp["cu_seqlens"], inp["has_init_conv"], 1, 2)
    args = (y, inp["alpha"], inp["beta"], inp["z"], inp["norm_w"], inp["state"], inp["slot_idx"],
            inp["cu_seqlens"], inp["has_init_state"], 1, 2)
    o_tok, s_tok, r_tok = orc.prefill(*args, chunk=0, want_raw=True)
    o_chk, s_chk, r_chk = orc.prefill(*args, chunk=chunk, want_raw=True)
    np.testing.assert_allclose(r_chk, r_tok, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(s_chk, s_tok, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(o_chk, o_tok, rtol=1e-10, atol=1e-10)


# ------------------------------------------------------------------ P8
def _conv_then_prefill(orc, inp, x, alpha, beta, z, cs, st, has_init, round_act):
    n = x.shape[0]
    cu = [0, n]
    slot = [0]
    y, cs2 = orc.conv_fwd(x, inp["conv_w"], cs, slot, cu, [has_init], inp["Hk"], inp["Hv"])
    if round_act:
        y = orc.round_bf16(y)
    out, st2 = orc.prefill(y, alpha, beta, z, inp["norm_w"], st, slot, cu, [has_init],
                           inp["Hk"], inp["Hv"])
    return out, cs2, st2


def _one_seq(n, seed):
    inp = syn.prefill_inputs([n], 2, 4, "bf16", seed=seed, init_mask=np.array([1]),
                             slot_perm=False, n_slots=1)
    return inp


def test_p8_split_prefill_equals_one_prefill(orc):
    n, cut = 23, 10
    inp = _one_seq(n, 71)
    x, a, b, z = inp["x"], inp["alpha"], inp["beta"], inp["z"]
    o_full, cs_full, st_full = _conv_then_prefill(orc, inp, x, a, b, z, inp["conv_state"],
                                                  inp["state"], 1, True)
    o1, cs1, st1 = _conv_then_prefill(orc, inp, x[:cut], a[:cut], b[:cut], z[:cut],
                                      inp["conv_state"], inp["state"], 1, True)
    o2, cs2, st2 = _conv_then_prefill(orc, inp, x[cut:], a[cut:], b[cut:], z[cut:],
                                      cs1, st1, 1, True)
    assert np.array_equal(np.concatenate([o1, o2]), o_full)
    assert np.array_equal(cs2, cs_full)
    assert np.array_equal(st2, st_full)


@pytest.mark.parametrize("T,ra", [(1, False), (3, False), (8, False), (3, True), (8, True)])
def test_p8_prefill_then_verify_equals_longer_prefill(orc, T, ra):
    """ra: the activations are rounded to bfloat16 on every side (stored rows)
    or on none (kept on chip); the identity holds bitwise either way."""
    n = 13
    inp = _one_seq(n + T, 72 + T)
    x, a, b, z = inp["x"], inp["alpha"], inp["beta"], inp["z"]
    Hk, Hv = inp["Hk"], inp["Hv"]
    o_full, cs_full, st_full = _conv_then_prefill(orc, inp, x, a, b, z, inp["conv_state"],
                                                  inp["state"], 1, ra)
    _, cs1, st1 = _conv_then_prefill(orc, inp, x[:n], a[:n], b[:n], z[:n],
                                     inp["conv_state"], inp["state"], 1, ra)
    out, _, cs_v, st_v = orc.verify(x[None, n:], inp["conv_w"], cs1, st1, a[None, n:],
                                    b[None, n:], z[None, n:], inp["norm_w"], [0], Hk, Hv,
                                    round_act=ra)
    assert np.array_equal(out[0], o_full[n:])
    assert np.array_equal(cs_v, cs1) and np.array_equal(st_v, st1)     # verify is read-only
    # commit of every draft token lands on the longer prefill's states
    for kind in ("commit", "commit_all"):
        if kind == "commit":
            cs_c, st_c = orc.commit(x[None, n:], a[None, n:], b[None, n:], inp["conv_w"], cs1, st1,
                                    [0], [T], Hk, Hv, round_act=ra)
        else:
            _, _, cs_c, st_c = orc.verify(x[None, n:], inp["conv_w"], cs1, st1, a[None, n:],
                                          b[None, n:], z[None, n:], inp["norm_w"], [0], Hk, Hv,
                                          commit_all=True, round_act=ra)
        assert np.array_equal(cs_c, cs_full)
        assert np.array_equal(st_c, st_full)


@pytest.mark.parametrize("n_keep,ra", [(0, False), (1, False), (2, False), (3, False),
                                        (5, False), (8, False), (2, True), (8, True)])
def test_p8_commit_equals_prefill_of_accepted_prefix(orc, n_keep, ra):
    T, n = 8, 9
    inp = _one_seq(n + T, 80 + n_keep)
    x, a, b, z = inp["x"], inp["alpha"], inp["beta"], inp["z"]
    Hk, Hv = inp["Hk"], inp["Hv"]
    _, cs1, st1 = _conv_then_prefill(orc, inp, x[:n], a[:n], b[:n], z[:n],
                                     inp["conv_state"], inp["state"], 1, ra)
    cs_c, st_c = orc.commit(x[None, n:], a[None, n:], b[None, n:], inp["conv_w"], cs1, st1, [0],
                            [n_keep], Hk, Hv, round_act=ra)
    if n_keep == 0:
        assert np.array_equal(cs_c, cs1) and np.array_equal(st_c, st1)
        return
    m = n + n_keep
    _, cs_p, st_p = _conv_then_prefill(orc, inp, x[:m], a[:m], b[:m], z[:m],
                                       inp["conv_state"], inp["state"], 1, ra)
    assert np.array_equal(cs_c, cs_p)
    assert np.array_equal(st_c, st_p)


@pytest.mark.parametrize("k,ra", [(0, False), (2, False), (6, False), (2, True)])
def test_p8_commit_then_next_verify_equals_longer_prefill(orc, k, ra):
    """Two verify windows of one sequence: the first window's k accepted drafts
    committed, then the second window's drafts verified, equal one prefill over
    the history, the accepted drafts and the new drafts (the rejected drafts of
    the first window leave no trace). This is the meaning of folding a window's
    commit into the next window's verify."""
    n, Tp, T = 9, 6, 4
    inp = _one_seq(n + Tp + T, 95 + k)
    x, a, b, z = inp["x"], inp["alpha"], inp["beta"], inp["z"]
    Hk, Hv = inp["Hk"], inp["Hv"]
    _, cs1, st1 = _conv_then_prefill(orc, inp, x[:n], a[:n], b[:n], z[:n],
                                     inp["conv_state"], inp["state"], 1, ra)
    w1 = slice(n, n + Tp)                                   # first window's drafts
    w2 = slice(n + Tp, n + Tp + T)                          # second window's drafts
    cs2, st2 = orc.commit(x[None, w1], a[None, w1], b[None, w1], inp["conv_w"], cs1, st1, [0], [k],
                          Hk, Hv, round_act=ra)
    out, _, _, _ = orc.verify(x[None, w2], inp["conv_w"], cs2, st2, a[None, w2], b[None, w2],
                              z[None, w2], inp["norm_w"], [0], Hk, Hv, round_act=ra)
    keep = np.r_[0:n + k, n + Tp:n + Tp + T]                # history ++ accepted ++ new drafts
    o_full, _, _ = _conv_then_prefill(orc, inp, x[keep], a[keep], b[keep], z[keep],
                                      inp["conv_state"], inp["state"], 1, ra)
    assert np.array_equal(out[0], o_full[n + k:])


def test_p8_commit_rejects_out_of_range_n_keep(orc):
    inp = syn.verify_inputs(3, 4, 1, 1, "f32", seed=90)
    cs, st = orc.commit(inp["x"], inp["alpha"], inp["beta"], inp["conv_w"], inp["conv_state"],
                        inp["state"], inp["slot_idx"], [5, -1, 0], 1, 1)
    assert np.array_equal(cs, inp["conv_state"].astype(np.float64))
    assert np.array_equal(st, inp["state"].astype(np.float64))


# ------------------------------------------------------------------ P9
@pytest.mark.parametrize("c", [0.75, -3.0, 1e-2])
def test_p9_rmsnorm_constant_vector(orc, c):
    eps = 1e-6
    o = np.full(D, c)
    out = orc.gated_rmsnorm(o, np.full(D, 40.0), np.ones(D), eps=eps)
    want = 40.0 * math.copysign(1.0, c) / math.sqrt(1.0 + eps / (c * c))
    np.testing.assert_allclose(out, want, rtol=1e-14)
    assert np.all(orc.gated_rmsnorm(o, np.zeros(D), np.ones(D)) == 0)


def test_p9_rmsnorm_weight_and_gate_are_elementwise(orc):
    rng = np.random.default_rng(95)
    o = rng.standard_normal(D)
    z = rng.standard_normal(D)
    w = rng.standard_normal(D)
    base = orc.gated_rmsnorm(o, np.full(D, 40.0), np.ones(D)) / 40.0
    rms = math.sqrt(sum(v * v for v in o) / D + 1e-6)
    np.testing.assert_allclose(base, o / rms, rtol=1e-13)
    out = orc.gated_rmsnorm(o, z, w)
    np.testing.assert_allclose(out, o / rms * w * z / (1 + np.exp(-z)), rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------------ P10
def test_p10_float_against_double(orc):
    inp = syn.workload_prefill("tiny-f32")
    args = (inp["x"], inp["conv_w"], inp["conv_state"], inp["slot_idx"], inp["cu_seqlens"],
            inp["has_init_conv"], inp["Hk"], inp["Hv"])
    y64, _ = orc.conv_fwd(*args, prec="f64")
    y32, _ = orc.conv_fwd(*args, prec="f32")
    # pre-activations: error of the f32 sum against the conditioning of the
    # 4-term sum (sum of |w_j x_j|), 10x under the 1e-5 bound
    pre64, _ = orc.conv_fwd(*args, silu=False, l2norm=False, prec="f64")
    pre32, _ = orc.conv_fwd(*args, silu=False, l2norm=False, prec="f32")
    wa = np.abs(inp["conv_w"]).astype(np.float64)
    xa = np.abs(np.concatenate([inp["conv_state"][inp["slot_idx"][0]], inp["x"]]))
    cond = sum(wa[None, :, j] * xa[j:j + 64] for j in range(4))
    assert np.max(np.abs(pre32 - pre64) / cond) < 1e-6
    # normalised activations (|y| <= 1): absolute error 10x under 1e-5
    assert np.max(np.abs(y32 - y64)) < 1e-6
    pa = (inp["alpha"], inp["beta"], inp["z"], inp["norm_w"], inp["state"], inp["slot_idx"],
          inp["cu_seqlens"], inp["has_init_state"], inp["Hk"], inp["Hv"])
    o64, s64 = orc.prefill(y64, *pa, prec="f64")
    o32, s32 = orc.prefill(y64.astype(np.float32), *pa, prec="f32")
    slot = inp["slot_idx"][0]
    for h in range(inp["Hv"]):
        fro = np.linalg.norm(s32[slot, h] - s64[slot, h]) / np.linalg.norm(s64[slot, h])
        assert fro < 1e-5
    assert np.max(np.abs(o32 - o64)) < 2e-3                  # 10x under the bf16 2e-2 bound
    # f32 recurrence outputs are held to 1e-4 x max(1, |ref|); stay 10x under it
    assert np.max(np.abs(o32 - o64) / np.maximum(1.0, np.abs(o64))) < 1e-5


# ------------------------------------------------------------------ BF
def test_bf16_rounding_matches_torch(orc):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(99)
    v = np.concatenate([rng.standard_normal(5000).astype(np.float32) * 100,
                        np.float32([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 3e-39])])
    want = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(orc.round_bf16(v, prec="f32"), want)
    assert np.array_equal(orc.round_bf16(v.astype(np.float64)), want.astype(np.float64))
    assert np.array_equal(syn.bf16_bits_to_f32(syn.f32_to_bf16_bits(v)), want)


# ------------------------------------------------------------------ GT
def test_gt_gates_closed_values(orc):
    """a = 0: softplus = ln 2, alpha = 1/2; b = 0: beta = 1/2 (exact)."""
    al, be = orc.gates(np.zeros(3), np.zeros(3))
    assert np.all(np.abs(al - 0.5) <= 2.0 ** -53) and np.all(be == 0.5)


def test_gt_gates_are_logistic_functions(orc):
    """exp(-log(1 + e^a)) = 1 / (1 + e^a) = expit(-a), and beta = expit(b): a sign
    slip, a dropped log1p or swapped outputs all break one of these."""
    special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(31)
    a = np.concatenate([np.linspace(-40.0, 40.0, 4001), 3.0 * rng.standard_normal(2000)])
    b = rng.permutation(a)
    al, be = orc.gates(a, b)
    np.testing.assert_allclose(al, special.expit(-a), rtol=1e-13, atol=0)
    np.testing.assert_allclose(be, special.expit(b), rtol=1e-13, atol=0)
    al2, be2 = orc.gates(-a, -b)
    np.testing.assert_allclose(al + al2, 1.0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(be + be2, 1.0, rtol=0, atol=1e-15)


def test_gt_gates_saturate_without_overflow(orc):
    for prec in ("f64", "f32"):
        a = np.array([-1000.0, -100.0, 100.0, 1000.0])
        al, be = orc.gates(a, a, prec=prec)
        assert np.all(np.isfinite(al)) and np.all(np.isfinite(be))
        assert al[0] == 1.0 and al[3] == 0.0 and be[0] == 0.0 and be[3] == 1.0
        assert 0.0 <= al[2] < 1e-40 and al[1] == 1.0


def test_gt_gates_float_against_double(orc):
    """The float instantiation (library expf / log1pf) within a few ulp of the
    double one; alpha's relative error grows with softplus(a) ~ |a| (its
    exponent's rounding)."""
    rng = np.random.default_rng(32)
    a = (3.0 * rng.standard_normal(20000)).astype(np.float32)
    b = (3.0 * rng.standard_normal(20000)).astype(np.float32)
    al32, be32 = orc.gates(a, b, prec="f32")
    al64, be64 = orc.gates(a.astype(np.float64), b.astype(np.float64))
    ulp = 2.0 ** -23
    assert np.all(np.abs(al32 - al64) <= al64 * ulp * (3.0 + 2.0 * np.abs(a)))
    assert np.all(np.abs(be32 - be64) <= be64 * ulp * 3.0)
