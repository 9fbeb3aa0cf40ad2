"""GPU parity of the gate step (alpha = exp(-softplus(a)), beta = sigmoid(b)).

"Strata PR #3226" tests a fused gate kernel against its multi-token form
bitwise. Here: gdn_gates against the oracle, and the GDN_GATES_RAW mode of the
prefill, verify, decode and commit kernels (the gate step applied to the raw
projections as they are read) bitwise against gdn_gates followed by the same
call on the activated gates, and against the oracle."""
import numpy as np
import pytest

from gated_deltanet_linear_12_gb300 import synthetic as syn
from tests.helpers import bits, check_bf16, check_f32_out, check_states, to_dev, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ULP = 2.0 ** -23
DENORM = 2.0 ** -147          # four steps of the float subnormal grid


@pytest.fixture(scope="module")
def G():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_linear_12_gb300 import gdn
    gdn.load()
    return gdn


def _check_gates(orc, a, b, al, be, what):
    """Within a few ulp of the exact gates; alpha's bound grows with softplus(a)
    ~ |a| (the rounding of its exponent), results in the subnormal range within
    four grid steps."""
    ra, rb = orc.gates(a.astype(np.float64), b.astype(np.float64))
    al, be = al.astype(np.float64), be.astype(np.float64)
    assert np.all(np.isfinite(al)) and np.all(np.isfinite(be)), what
    err_a = np.abs(al - ra) - (ra * ULP * (6.0 + 2.0 * np.abs(a.astype(np.float64))) + DENORM)
    err_b = np.abs(be - rb) - (rb * ULP * 6.0 + DENORM)
    assert err_a.max() <= 0, f"{what}: alpha out of bound at {np.argmax(err_a)}"
    assert err_b.max() <= 0, f"{what}: beta out of bound at {np.argmax(err_b)}"


def _gates_dev(G, cfg, a, b):
    al, be = torch.empty_like(a), torch.empty_like(b)
    G.gdn_gates(cfg, a, b, al, be)
    return al, be


def test_gates_kernel_against_oracle(G, orc):
    """Ragged count (tail past the 16-byte groups), saturating values, the
    unaligned path and in place: every route gives the same bits."""
    n_tok, Hv = 37, 6
    rng = np.random.default_rng(610)
    a = (3.0 * rng.standard_normal((n_tok, Hv))).astype(np.float32)
    b = (3.0 * rng.standard_normal((n_tok, Hv))).astype(np.float32)
    ext = np.array([-1000, -104, -100, -88, -20, -1e-3, 0, 1e-3, 20, 88, 100, 104, 1000], np.float32)
    a.flat[:ext.size] = ext
    b.flat[-ext.size:] = ext
    cfg = G.make_config(1, Hv, torch.bfloat16, 1)
    da, db = to_dev(a), to_dev(b)
    al, be = _gates_dev(G, cfg, da, db)
    torch.cuda.synchronize()
    _check_gates(orc, a, b, to_np(al), to_np(be), "gdn_gates")
    # unaligned path: the same values one float into a buffer
    fa = torch.zeros(a.size + 1, device="cuda")
    fb = torch.zeros(a.size + 1, device="cuda")
    fa[1:] = da.flatten()
    fb[1:] = db.flatten()
    ua, ub = fa[1:].view(n_tok, Hv), fb[1:].view(n_tok, Hv)
    oa, ob = torch.zeros(a.size + 1, device="cuda"), torch.zeros(a.size + 1, device="cuda")
    G.gdn_gates(cfg, ua, ub, oa[1:].view(n_tok, Hv), ob[1:].view(n_tok, Hv))
    # in place
    ia, ib = da.clone(), db.clone()
    G.gdn_gates(cfg, ia, ib, ia, ib)
    torch.cuda.synchronize()
    for x, y in ((oa[1:].view(n_tok, Hv), ob[1:].view(n_tok, Hv)), (ia, ib)):
        assert np.array_equal(bits(x), bits(al)) and np.array_equal(bits(y), bits(be))
    assert float(oa[0]) == 0.0 and float(ob[0]) == 0.0, "nothing written before the range"


def test_gates_empty_is_a_no_op(G):
    cfg = G.make_config(1, 4, torch.bfloat16, 1)
    e = torch.empty(0, 4, device="cuda")
    G.gdn_gates(cfg, e, e.clone(), e.clone(), e.clone())


# ------------------------------------------------------------------ prefill
def _post_conv(orc, inp):
    """Post-conv rows as stored: the double oracle's values rounded to the
    activation dtype (an input of both sides)."""
    y, _ = orc.conv_fwd(inp["x"], inp["conv_w"], inp["conv_state"], inp["slot_idx"],
                        inp["cu_seqlens"], inp["has_init_conv"], inp["Hk"], inp["Hv"])
    if inp["act"] == "bf16":
        y = orc.round_bf16(y)
    return syn.to_act(y.astype(np.float32), inp["act"])


def _prefill(G, inp, qkv, al, be, gates):
    act = torch.bfloat16 if inp["act"] == "bf16" else torch.float32
    S = to_dev(inp["state"])
    out = torch.zeros(inp["n_tok"], inp["Hv"] * 128, dtype=act, device="cuda")
    cfg = G.make_config(inp["Hk"], inp["Hv"], act, S.shape[0], gates=gates)
    G.gdn_delta_prefill(cfg, to_dev(qkv), al, be, to_dev(inp["z"]), to_dev(inp["norm_w"]), out, S,
                        to_dev(inp["slot_idx"]), to_dev(inp["cu_seqlens"]),
                        to_dev(inp["has_init_state"]))
    torch.cuda.synchronize()
    return out, S


@pytest.mark.parametrize("act", ["bf16", "f32"])
def test_prefill_raw_gates(G, orc, act):
    """Partial last chunks (70, 129, 5 tokens): the padded tokens keep beta = 0."""
    inp = syn.prefill_inputs([70, 129, 5], 2, 4, act, seed=620, init_mask=np.array([1, 0, 1]),
                             gate_form="raw")
    qkv = _post_conv(orc, inp)
    a, b = to_dev(inp["alpha"]), to_dev(inp["beta"])
    out_r, S_r = _prefill(G, inp, qkv, a, b, G.GDN_GATES_RAW)
    cfg = G.make_config(inp["Hk"], inp["Hv"], torch.float32, 1)
    al, be = _gates_dev(G, cfg, a, b)
    out_a, S_a = _prefill(G, inp, qkv, al, be, G.GDN_GATES_ACTIVATED)
    assert np.array_equal(bits(out_r), bits(out_a)), "raw gates == gdn_gates + prefill (bitwise)"
    assert np.array_equal(bits(S_r), bits(S_a))
    ra, rb = orc.gates(inp["alpha"], inp["beta"])
    ro, rs = orc.prefill(qkv, ra, rb, inp["z"], inp["norm_w"], inp["state"], inp["slot_idx"],
                         inp["cu_seqlens"], inp["has_init_state"], inp["Hk"], inp["Hv"])
    if act == "bf16":
        check_bf16(to_np(out_r), ro, what="prefill raw gates out")
    else:
        check_f32_out(to_np(out_r), ro, 1e-4, "prefill raw gates out")
    check_states(to_np(S_r), rs, [int(s) for s in inp["slot_idx"]], 1e-4, "prefill raw gates state")


# ------------------------------------------------------------------ verify / decode / commit
class Win:
    """Device copies of one layer's verify inputs; alpha / beta as given."""

    def __init__(self, inp, al, be):
        self.inp = inp
        self.act = torch.bfloat16 if inp["act"] == "bf16" else torch.float32
        self.x, self.conv_w = to_dev(inp["x"]), to_dev(inp["conv_w"])
        self.cs, self.S = to_dev(inp["conv_state"]), to_dev(inp["state"])
        self.al, self.be = al, be
        self.z, self.norm_w, self.slot = to_dev(inp["z"]), to_dev(inp["norm_w"]), to_dev(inp["slot_idx"])
        B, T, Hv = inp["B"], inp["T"], inp["Hv"]
        self.out = torch.zeros(B, T, Hv * 128, dtype=self.act, device="cuda")
        self.pc = torch.zeros(B, T, inp["C"], dtype=self.act, device="cuda")

    def cfg(self, G, gates):
        return G.make_config(self.inp["Hk"], self.inp["Hv"], self.act, self.S.shape[0], gates=gates)

    def verify(self, G, gates, commit_all=False):
        G.gdn_verify_step(self.cfg(G, gates), self.x, self.conv_w, self.cs, self.S, self.al, self.be,
                          self.z, self.norm_w, self.out, self.slot, commit_all=commit_all,
                          postconv_out=self.pc)

    def view(self):
        return dict(x=self.x, alpha=self.al, beta=self.be, conv_w=self.conv_w, conv_state=self.cs,
                    state=self.S)


def _pair(G, inp):
    """(raw window, activated window) over the same inputs."""
    a, b = to_dev(inp["alpha"]), to_dev(inp["beta"])
    al, be = _gates_dev(G, G.make_config(inp["Hk"], inp["Hv"], torch.float32, 1), a, b)
    return Win(inp, a, b), Win(inp, al, be)


@pytest.mark.parametrize("T,act,commit_all", [(3, "bf16", False), (8, "bf16", False),
                                              (5, "f32", False), (1, "bf16", True), (4, "bf16", True)])
def test_verify_and_decode_raw_gates(G, orc, T, act, commit_all):
    inp = syn.verify_inputs(6, T, 2, 4, act, seed=630 + T, pad_slots=1, gate_form="raw")
    R, A = _pair(G, inp)
    R.verify(G, G.GDN_GATES_RAW, commit_all)
    A.verify(G, G.GDN_GATES_ACTIVATED, commit_all)
    torch.cuda.synchronize()
    for x, y in ((R.out, A.out), (R.pc, A.pc), (R.S, A.S), (R.cs, A.cs)):
        assert np.array_equal(bits(x), bits(y)), "raw gates == gdn_gates + verify (bitwise)"
    ra, rb = orc.gates(inp["alpha"], inp["beta"])
    out, _, cs, st = orc.verify(inp["x"], inp["conv_w"], inp["conv_state"], inp["state"], ra, rb,
                                inp["z"], inp["norm_w"], inp["slot_idx"], inp["Hk"], inp["Hv"],
                                commit_all=commit_all)
    if act == "bf16":
        check_bf16(to_np(R.out), out, what=f"verify raw gates T={T}")
    else:
        check_f32_out(to_np(R.out), out, 1e-4, f"verify raw gates f32 T={T}")
    if commit_all:
        assert np.array_equal(to_np(R.cs), cs)
        used = [int(s) for s in inp["slot_idx"] if s >= 0]
        check_states(to_np(R.S), st, used, 1e-4, "decode raw gates state")


@pytest.mark.parametrize("T", [2, 7])
def test_commit_raw_gates(G, orc, T):
    nl = 2
    inps = [syn.verify_inputs(5, T, 2, 4, "bf16", seed=650 + 10 * T + l, gate_form="raw")
            for l in range(nl)]
    n_keep = inps[0]["n_keep"].copy()
    n_keep[0], n_keep[1] = 0, T
    for inp in inps:
        inp["slot_idx"] = inps[0]["slot_idx"]
    pairs = [_pair(G, inp) for inp in inps]
    nk = to_dev(n_keep)
    for k, gates in ((0, G.GDN_GATES_RAW), (1, G.GDN_GATES_ACTIVATED)):
        wins = [p[k] for p in pairs]
        views = G.make_layer_views([w.view() for w in wins], "cuda")
        G.gdn_commit_layers(wins[0].cfg(G, gates), views, nl, wins[0].slot, nk, T)
    torch.cuda.synchronize()
    for (R, A), inp in zip(pairs, inps):
        assert np.array_equal(bits(R.S), bits(A.S)), "raw gates == gdn_gates + commit (bitwise)"
        assert np.array_equal(bits(R.cs), bits(A.cs))
        ra, rb = orc.gates(inp["alpha"], inp["beta"])
        cs, st = orc.commit(inp["x"], ra, rb, inp["conv_w"], inp["conv_state"], inp["state"],
                            inp["slot_idx"], n_keep, 2, 4)
        assert np.array_equal(to_np(R.cs), cs), "conv_state commit must be bit-exact"
        check_states(to_np(R.S), st, range(st.shape[0]), 1e-4, "commit raw gates state")


# ------------------------------------------------------------------ bf16 gate arrays
def _bf16(a):
    return syn.f32_to_bf16_bits(np.asarray(a, np.float32))


def test_gates_kernel_bf16_io(G, orc):
    """gdn_gates with bfloat16 a, b, alpha, beta: the results are the f32 gates
    of the widened inputs rounded to nearest even; the f32-output arm (f32
    arrays holding the same bf16 values) gives those unrounded gates."""
    n_tok, Hv = 41, 5
    rng = np.random.default_rng(615)
    a16 = _bf16(3.0 * rng.standard_normal((n_tok, Hv)))
    b16 = _bf16(3.0 * rng.standard_normal((n_tok, Hv)))
    a32, b32 = syn.bf16_bits_to_f32(a16), syn.bf16_bits_to_f32(b16)      # exact widening
    cfg16 = G.make_config(1, Hv, torch.bfloat16, 1, gate_dtype=torch.bfloat16)
    al16, be16 = _gates_dev(G, cfg16, to_dev(a16), to_dev(b16))
    cfg32 = G.make_config(1, Hv, torch.bfloat16, 1)
    al32, be32 = _gates_dev(G, cfg32, to_dev(a32), to_dev(b32))
    torch.cuda.synchronize()
    _check_gates(orc, a32, b32, to_np(al32), to_np(be32), "gdn_gates f32 arm of bf16 inputs")
    ra, rb = orc.gates(a32.astype(np.float64), b32.astype(np.float64))
    check_bf16(to_np(al16), ra, atol=0.0, what="bf16 alpha")
    check_bf16(to_np(be16), rb, atol=0.0, what="bf16 beta")
    # bitwise: the bf16 results are the f32 results rounded
    assert np.array_equal(bits(al16), _bf16(to_np(al32)).view(np.int16))
    assert np.array_equal(bits(be16), _bf16(to_np(be32)).view(np.int16))


@pytest.mark.parametrize("gates", ["raw", "activated"])
@pytest.mark.parametrize("out_f32", [False, True])
def test_prefill_bf16_gate_arrays(G, orc, gates, out_f32):
    """bf16 gate arrays (raw a, b or activated alpha, beta) in the tensor-core
    prefill: bitwise equal to the f32 arrays holding the same values, and
    against the oracle on the widened gates, with an f32-output arm."""
    inp = syn.prefill_inputs([70, 129, 5], 2, 4, "bf16", seed=625, init_mask=np.array([1, 0, 1]),
                             gate_form="raw" if gates == "raw" else "softplus")
    qkv = _post_conv(orc, inp)
    g16 = (_bf16(inp["alpha"]), _bf16(inp["beta"]))
    g32 = tuple(syn.bf16_bits_to_f32(g) for g in g16)
    mode = G.GDN_GATES_RAW if gates == "raw" else G.GDN_GATES_ACTIVATED
    res = []
    for gd, (al, be) in ((torch.bfloat16, g16), (torch.float32, g32)):
        S = to_dev(inp["state"])
        out = torch.zeros(inp["n_tok"], inp["Hv"] * 128, dtype=torch.float32 if out_f32 else torch.bfloat16,
                          device="cuda")
        cfg = G.make_config(inp["Hk"], inp["Hv"], torch.bfloat16, S.shape[0], gates=mode, gate_dtype=gd,
                            out_f32=out_f32)
        G.gdn_delta_prefill(cfg, to_dev(qkv), to_dev(al), to_dev(be), to_dev(inp["z"]), to_dev(inp["norm_w"]),
                            out, S, to_dev(inp["slot_idx"]), to_dev(inp["cu_seqlens"]),
                            to_dev(inp["has_init_state"]))
        res.append((out, S))
    torch.cuda.synchronize()
    assert np.array_equal(bits(res[0][0]), bits(res[1][0])), "bf16 gates == the same values in f32 (bitwise)"
    assert np.array_equal(bits(res[0][1]), bits(res[1][1]))
    ra, rb = (orc.gates(*g32) if gates == "raw" else g32)
    ro, rs = orc.prefill(qkv, ra, rb, inp["z"], inp["norm_w"], inp["state"], inp["slot_idx"],
                         inp["cu_seqlens"], inp["has_init_state"], inp["Hk"], inp["Hv"])
    if out_f32:
        check_f32_out(to_np(res[0][0]), ro, 1e-4, "prefill bf16 gates, f32 out")
    else:
        check_bf16(to_np(res[0][0]), ro, what="prefill bf16 gates out")
    check_states(to_np(res[0][1]), rs, [int(s) for s in inp["slot_idx"]], 1e-4, "prefill bf16 gates state")


@pytest.mark.parametrize("T,commit_all", [(3, False), (8, False), (1, True), (5, True)])
def test_verify_bf16_gate_arrays(G, orc, T, commit_all):
    """bf16 raw gates in verify / decode and the batched commit: bitwise equal to
    f32 arrays holding the same values, and against the oracle."""
    inp = syn.verify_inputs(5, T, 2, 4, "bf16", seed=640 + T, pad_slots=1, gate_form="raw")
    a16, b16 = _bf16(inp["alpha"]), _bf16(inp["beta"])
    a32, b32 = syn.bf16_bits_to_f32(a16), syn.bf16_bits_to_f32(b16)
    wins = []
    for gd, (a, b) in ((torch.bfloat16, (a16, b16)), (torch.float32, (a32, b32))):
        w = Win(inp, to_dev(a), to_dev(b))
        cfg = G.make_config(2, 4, torch.bfloat16, w.S.shape[0], gates=G.GDN_GATES_RAW, gate_dtype=gd)
        G.gdn_verify_step(cfg, w.x, w.conv_w, w.cs, w.S, w.al, w.be, w.z, w.norm_w, w.out, w.slot,
                          commit_all=commit_all)
        if not commit_all:
            views = G.make_layer_views([w.view()], "cuda")
            G.gdn_commit_layers(cfg, views, 1, w.slot, to_dev(inp["n_keep"]), T)
        wins.append(w)
    torch.cuda.synchronize()
    for x, y in ((wins[0].out, wins[1].out), (wins[0].S, wins[1].S), (wins[0].cs, wins[1].cs)):
        assert np.array_equal(bits(x), bits(y)), "bf16 gates == the same values in f32 (bitwise)"
    ra, rb = orc.gates(a32, b32)
    out, _, cs, st = orc.verify(inp["x"], inp["conv_w"], inp["conv_state"], inp["state"], ra, rb,
                                inp["z"], inp["norm_w"], inp["slot_idx"], 2, 4, commit_all=commit_all)
    check_bf16(to_np(wins[0].out), out, what=f"verify bf16 gates T={T}")
    if not commit_all:
        cs, st = orc.commit(inp["x"], ra, rb, inp["conv_w"], inp["conv_state"], inp["state"],
                            inp["slot_idx"], inp["n_keep"], 2, 4)
    assert np.array_equal(to_np(wins[0].cs), cs)
    used = [int(s) for s in inp["slot_idx"] if s >= 0]
    check_states(to_np(wins[0].S), st, used, 1e-4, "bf16 gates state")
