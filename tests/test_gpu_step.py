"""GPU parity of speculative verify, decode (verify with every token accepted)
and the batched accepted-prefix commit, against the CPU oracle and against
each other (bitwise), through the C ABI."""
import numpy as np
import pytest

from gated_deltanet_linear_12_gb300 import synthetic as syn
from tests.helpers import Canary, bits, check_bf16, check_f32_out, check_states, to_dev, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def G():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_linear_12_gb300 import gdn
    gdn.load()
    return gdn


class Layer:
    """Device copies of one layer's verify inputs and pools."""

    def __init__(self, inp):
        self.inp = inp
        self.act = torch.bfloat16 if inp["act"] == "bf16" else torch.float32
        self.guard = Canary()                      # pools, drafts and outputs between NaN bands
        self.x = self.guard.wrap(to_dev(inp["x"]))
        self.conv_w = to_dev(inp["conv_w"])
        self.cs = self.guard.wrap(to_dev(inp["conv_state"]))
        self.S = self.guard.wrap(to_dev(inp["state"]))
        self.alpha = to_dev(inp["alpha"])
        self.beta = to_dev(inp["beta"])
        self.z = to_dev(inp["z"])
        self.norm_w = to_dev(inp["norm_w"])
        self.slot = to_dev(inp["slot_idx"])
        B, T, Hv = inp["B"], inp["T"], inp["Hv"]
        self.out = self.guard.wrap(torch.zeros(B, T, Hv * 128, dtype=self.act, device="cuda"))
        self.pc = self.guard.wrap(torch.zeros(B, T, inp["C"], dtype=self.act, device="cuda"))

    def cfg(self, G, dev_err=None):
        return G.make_config(self.inp["Hk"], self.inp["Hv"], self.act, self.S.shape[0],
                             dev_err=dev_err)

    def verify(self, G, commit_all=False, dev_err=None):
        G.gdn_verify_step(self.cfg(G, dev_err), self.x, self.conv_w, self.cs, self.S, self.alpha,
                          self.beta, self.z, self.norm_w, self.out, self.slot,
                          commit_all=commit_all, postconv_out=self.pc)

    def view(self):
        return dict(x=self.x, alpha=self.alpha, beta=self.beta, conv_w=self.conv_w,
                    conv_state=self.cs, state=self.S)


def _oracle_verify(orc, inp, commit_all=False):
    """Oracle verify in double: the plain conv, SiLU and norms, the activations
    unrounded into the token-by-token recurrence (the fused kernels keep them
    on chip), then the gated RMSNorm."""
    return orc.verify(inp["x"], inp["conv_w"], inp["conv_state"], inp["state"], inp["alpha"],
                      inp["beta"], inp["z"], inp["norm_w"], inp["slot_idx"], inp["Hk"], inp["Hv"],
                      commit_all=commit_all)


def _check_postconv(pc_gpu, pc_ref, act, what="post-conv"):
    """The stored post-conv copy against the double oracle's unrounded values."""
    if act == "bf16":
        check_bf16(to_np(pc_gpu), pc_ref, what=what)
    else:
        check_f32_out(to_np(pc_gpu), pc_ref, 1e-5, what)


def _used_slots(inp):
    return [int(s) for s in inp["slot_idx"] if s >= 0]


@pytest.mark.parametrize("T", range(1, 9))                 # every compiled variant
def test_verify_bf16(G, orc, T):
    inp = syn.verify_inputs(6, T, 2, 4, "bf16", seed=200 + T, pad_slots=1)
    L = Layer(inp)
    L.verify(G)
    torch.cuda.synchronize()
    out, pc, cs, st = _oracle_verify(orc, inp)
    check_bf16(to_np(L.out), out, what=f"verify out T={T}")
    _check_postconv(L.pc[:5], pc[:5], "bf16")
    # verify is read-only
    assert np.array_equal(bits(L.cs), inp["conv_state"].view(np.int16))
    assert np.array_equal(bits(L.S), inp["state"].view(np.int32))
    assert np.all(to_np(L.out)[5] == 0), "padding entry must not be written"
    L.guard.check(f"verify T={T}")


@pytest.mark.parametrize("T", range(1, 9))                 # every compiled variant
def test_verify_f32_arm(G, orc, T):
    inp = syn.verify_inputs(3, T, 1, 2, "f32", seed=210 + T)
    L = Layer(inp)
    L.verify(G)
    torch.cuda.synchronize()
    out, pc, _, _ = _oracle_verify(orc, inp)
    check_f32_out(to_np(L.out), out, 1e-4, f"verify f32 out T={T}")


# Tolerance of f32 outputs computed with the tensor core's tf32 products (bf16
# activations, T >= 5): the state and the f32 activations enter with 10 explicit
# mantissa bits, a relative error up to 2^-10 per operand (truncation); the
# products and dot products then carry about 2^-9 of the sum of |terms| and the
# normalised outputs (RMS 1 before the weight and gate) an error near 2^-9.
TF32_OUT_TOL = 4e-3


@pytest.mark.parametrize("T", range(1, 9))
def test_verify_bf16_act_f32_out(G, orc, T):
    """The f32-output arm of the bf16 verify: the CUDA-core variants (T <= 4) at
    the f32 recurrence tolerance, the tensor-core variant (T >= 5) at the bound
    of its tf32 products, which stays 5x under the bf16 output tolerance."""
    inp = syn.verify_inputs(6, T, 2, 4, "bf16", seed=230 + T, pad_slots=1)
    L = Layer(inp)
    L.out = torch.zeros(inp["B"], T, inp["Hv"] * 128, dtype=torch.float32, device="cuda")
    cfg = G.make_config(2, 4, torch.bfloat16, L.S.shape[0], out_f32=True)
    G.gdn_verify_step(cfg, L.x, L.conv_w, L.cs, L.S, L.alpha, L.beta, L.z, L.norm_w, L.out, L.slot,
                      postconv_out=L.pc)
    torch.cuda.synchronize()
    out, pc, _, _ = _oracle_verify(orc, inp)
    tol = 1e-4 if T <= 4 else TF32_OUT_TOL
    check_f32_out(to_np(L.out)[:5], out[:5], tol, f"verify bf16 act, f32 out, T={T}")
    assert np.all(to_np(L.out)[5] == 0), "padding entry must not be written"
    assert np.array_equal(bits(L.S), inp["state"].view(np.int32))


@pytest.mark.parametrize("T", [1, 8])
def test_decode_bf16_act_f32_out(G, orc, T):
    """Decode (commit-all) with f32 outputs: CUDA-core products at every T."""
    inp = syn.verify_inputs(4, T, 2, 4, "bf16", seed=240 + T)
    L = Layer(inp)
    L.out = torch.zeros(inp["B"], T, inp["Hv"] * 128, dtype=torch.float32, device="cuda")
    cfg = G.make_config(2, 4, torch.bfloat16, L.S.shape[0], out_f32=True)
    G.gdn_verify_step(cfg, L.x, L.conv_w, L.cs, L.S, L.alpha, L.beta, L.z, L.norm_w, L.out, L.slot,
                      commit_all=True)
    torch.cuda.synchronize()
    out, _, cs, st = _oracle_verify(orc, inp, commit_all=True)
    check_f32_out(to_np(L.out), out, 1e-4, f"decode f32 out T={T}")
    assert np.array_equal(to_np(L.cs), cs)
    check_states(to_np(L.S), st, _used_slots(inp), 1e-4, "decode f32-out state")


@pytest.mark.parametrize("T", [1, 3, 8])
def test_commit_all_equals_verify_then_commit_bitwise(G, orc, T):
    inp = syn.verify_inputs(5, T, 2, 4, "bf16", seed=220 + T)
    A = Layer(inp)
    A.verify(G, commit_all=True)
    Bl = Layer(inp)
    Bl.verify(G)
    views = G.make_layer_views([Bl.view()], "cuda")
    n_keep = torch.full((5,), T, dtype=torch.int32, device="cuda")
    G.gdn_commit_layers(Bl.cfg(G), views, 1, Bl.slot, n_keep, T)
    torch.cuda.synchronize()
    A.guard.check("decode")
    assert np.array_equal(bits(A.S), bits(Bl.S)), "decode == verify + commit(T), bitwise"
    assert np.array_equal(bits(A.cs), bits(Bl.cs))
    if T == 1:                       # same variant: outputs bitwise too
        assert np.array_equal(bits(A.out), bits(Bl.out))
    else:                            # verify uses the tensor cores: rounding only
        check_bf16(to_np(A.out), to_np(Bl.out), what="decode vs verify outputs")
    # and against the oracle
    out, _, cs, st = _oracle_verify(orc, inp, commit_all=True)
    check_bf16(to_np(A.out), out, what="decode out")
    assert np.array_equal(to_np(A.cs), cs), "conv_state commit must be bit-exact"
    check_states(to_np(A.S), st, range(st.shape[0]), 1e-4, "decode state")


@pytest.mark.parametrize("T", [2, 5, 8])
def test_commit_layers_against_oracle_and_per_layer(G, orc, T):
    nl = 3
    inps = [syn.verify_inputs(7, T, 2, 4, "bf16", seed=300 + 10 * T + l) for l in range(nl)]
    n_keep = syn.verify_inputs(7, T, 2, 4, "bf16", seed=399)["n_keep"]
    n_keep[0], n_keep[1] = 0, T                     # both ends always present
    for inp in inps:
        inp["n_keep"] = n_keep
        inp["slot_idx"] = inps[0]["slot_idx"]
    batched = [Layer(i) for i in inps]
    single = [Layer(i) for i in inps]
    nk = to_dev(n_keep)
    views = G.make_layer_views([l.view() for l in batched], "cuda")
    G.gdn_commit_layers(batched[0].cfg(G), views, nl, batched[0].slot, nk, T)
    for l in single:
        v1 = G.make_layer_views([l.view()], "cuda")
        G.gdn_commit_layers(l.cfg(G), v1, 1, l.slot, nk, T)
        torch.cuda.synchronize()
    torch.cuda.synchronize()
    for lb, ls, inp in zip(batched, single, inps):
        lb.guard.check("batched commit")
        assert np.array_equal(bits(lb.S), bits(ls.S)), "batched == per-layer commit (bitwise)"
        assert np.array_equal(bits(lb.cs), bits(ls.cs))
        cs, st = orc.commit(inp["x"], inp["alpha"], inp["beta"], inp["conv_w"], inp["conv_state"],
                            inp["state"], inp["slot_idx"], n_keep, 2, 4)
        assert np.array_equal(to_np(lb.cs), cs), "conv_state commit must be bit-exact"
        check_states(to_np(lb.S), st, range(st.shape[0]), 1e-4, "committed state")
        # slots with n_keep == 0 and slots nobody references stay bitwise untouched
        keep0 = [int(inp["slot_idx"][b]) for b in range(7) if n_keep[b] == 0]
        unused = sorted(set(range(inp["state"].shape[0])) - set(int(s) for s in inp["slot_idx"]))
        for sl in keep0 + unused:
            assert np.array_equal(bits(lb.S)[sl], inp["state"][sl].view(np.int32))
            assert np.array_equal(bits(lb.cs)[sl], inp["conv_state"][sl].view(np.int16))


def test_commit_bad_n_keep_and_slot_flag_errors(G):
    T = 4
    inp = syn.verify_inputs(4, T, 1, 2, "bf16", seed=410)
    L = Layer(inp)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    n_keep = torch.tensor([T + 1, 2, -1, 1], dtype=torch.int32, device="cuda")
    slots = inp["slot_idx"].copy()
    slots[3] = inp["state"].shape[0] + 7
    L.slot = to_dev(slots)
    views = G.make_layer_views([L.view()], "cuda")
    G.gdn_commit_layers(L.cfg(G, err), views, 1, L.slot, n_keep, T)
    torch.cuda.synchronize()
    e = int(err.item())
    assert e & G.GDN_DEVERR_NKEEP and e & G.GDN_DEVERR_SLOT
    S = bits(L.S)
    for b in (0, 2):                                  # skipped entries untouched
        sl = slots[b]
        assert np.array_equal(S[sl], inp["state"][sl].view(np.int32))
    assert not np.array_equal(S[slots[1]], inp["state"][slots[1]].view(np.int32))


@pytest.mark.parametrize("T", [1, 8])
def test_verify_group_of_three_v_heads(G, orc, T):
    """Hv/Hk = 3 (the 48-over-16 grouping of a larger model)."""
    inp = syn.verify_inputs(3, T, 2, 6, "bf16", seed=420 + T)
    L = Layer(inp)
    L.verify(G, commit_all=True)
    torch.cuda.synchronize()
    out, _, cs, st = _oracle_verify(orc, inp, commit_all=True)
    check_bf16(to_np(L.out), out, what="verify G=3")
    assert np.array_equal(to_np(L.cs), cs)
    check_states(to_np(L.S), st, _used_slots(inp), 1e-4, "state G=3")


@pytest.mark.parametrize("T", [1, 3, 5, 8])
def test_verify_window_geometry_48_v_heads(G, orc, T):
    """The verify window of "Strata PR #3226" ("Benchmark Evidence"): one sequence,
    Hk = 16, Hv = 48 (C = 10240), read-only verify then the commit of n tokens."""
    inp = syn.verify_inputs(1, T, 16, 48, "bf16", seed=440 + T, n_slots=2)
    L = Layer(inp)
    L.verify(G)
    torch.cuda.synchronize()
    out, pc, _, _ = _oracle_verify(orc, inp)
    check_bf16(to_np(L.out), out, what=f"verify Hv=48 T={T}")
    _check_postconv(L.pc, pc, "bf16")
    assert np.array_equal(bits(L.S), inp["state"].view(np.int32))
    L.verify(G, commit_all=True)
    torch.cuda.synchronize()
    out2, _, cs, st = _oracle_verify(orc, inp, commit_all=True)
    check_bf16(to_np(L.out), out2, what=f"decode Hv=48 T={T}")
    assert np.array_equal(to_np(L.cs), cs)
    check_states(to_np(L.S), st, _used_slots(inp), 1e-4, f"state Hv=48 T={T}")


@pytest.mark.parametrize("T,act", [(3, "bf16"), (8, "bf16"), (5, "f32")])
def test_verify_q_scale_and_eps(G, orc, T, act):
    """q_scale = d^-1/2 with an eps large enough that the output RMSNorm does not
    divide the scale away (eps also enters the q/k norms, on both sides)."""
    inp = syn.verify_inputs(4, T, 2, 4, act, seed=460 + T)
    L = Layer(inp)
    qs, eps = 128 ** -0.5, 0.05
    cfg = G.make_config(inp["Hk"], inp["Hv"], L.act, L.S.shape[0], q_scale=qs, eps=eps)
    G.gdn_verify_step(cfg, L.x, L.conv_w, L.cs, L.S, L.alpha, L.beta, L.z, L.norm_w, L.out, L.slot,
                      postconv_out=L.pc)
    torch.cuda.synchronize()
    out, pc, _, _ = orc.verify(inp["x"], inp["conv_w"], inp["conv_state"], inp["state"], inp["alpha"],
                               inp["beta"], inp["z"], inp["norm_w"], inp["slot_idx"], inp["Hk"],
                               inp["Hv"], q_scale=qs, eps=eps)
    _check_postconv(L.pc, pc, act)
    if act == "bf16":
        check_bf16(to_np(L.out), out, what=f"verify q_scale T={T}")
    else:
        check_f32_out(to_np(L.out), out, 1e-4, f"verify q_scale f32 T={T}")


def test_verify_postconv_matches_conv_fwd_bitwise(G):
    """The activations verify uses equal gdn_conv_fwd's on the same rows."""
    T = 6
    inp = syn.verify_inputs(2, T, 2, 4, "bf16", seed=430)
    L = Layer(inp)
    L.verify(G)
    C = inp["C"]
    x = L.x.reshape(2 * T, C)
    y = torch.empty_like(x)
    cs = to_dev(inp["conv_state"])
    cu = torch.tensor([0, T, 2 * T], dtype=torch.int32, device="cuda")
    hi = torch.ones(2, dtype=torch.uint8, device="cuda")
    G.gdn_conv_fwd(L.cfg(G), x, y, L.conv_w, cs, L.slot, cu, hi)
    torch.cuda.synchronize()
    assert np.array_equal(bits(y), bits(L.pc.reshape(2 * T, C)))
