"""GPU parity of the verify with the previous window's commit folded in
(gdn_verify_step_lazy): its committed conv_state and state are bitwise those of
gdn_commit_layers, its outputs match the oracle's commit-then-verify, and a
chain of windows leaves the same state bits as the verify / commit route."""
import numpy as np
import pytest

from gated_deltanet_linear_12_gb300 import synthetic as syn
from tests.helpers import bits, check_bf16, check_f32_out, check_states, to_dev, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

HK, HV = 2, 4


@pytest.fixture(scope="module")
def G():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_linear_12_gb300 import gdn
    gdn.load()
    return gdn


def _windows(B, Ts, act, seed, pad=1):
    """Inputs of consecutive windows of one layer: shared pools, weights and
    slots, fresh drafts, gates and z per window."""
    ws = [syn.verify_inputs(B, T, HK, HV, act, seed=seed + i, pad_slots=pad) for i, T in enumerate(Ts)]
    for w in ws[1:]:
        for k in ("slot_idx", "conv_state", "state", "conv_w", "norm_w"):
            w[k] = ws[0][k]
    for w in ws:
        w["n_keep"][0], w["n_keep"][1] = 0, w["T"]                # both ends present
    return ws


class Pools:
    def __init__(self, w):
        self.act = torch.bfloat16 if w["act"] == "bf16" else torch.float32
        self.cs, self.S = to_dev(w["conv_state"]), to_dev(w["state"])
        self.conv_w, self.norm_w, self.slot = to_dev(w["conv_w"]), to_dev(w["norm_w"]), to_dev(w["slot_idx"])

    def cfg(self, G, dev_err=None):
        return G.make_config(HK, HV, self.act, self.S.shape[0], dev_err=dev_err)

    def bufs(self, w):
        B, T = w["B"], w["T"]
        out = torch.zeros(B, T, HV * 128, dtype=self.act, device="cuda")
        pc = torch.zeros(B, T, w["C"], dtype=self.act, device="cuda")
        return out, pc

    def verify(self, G, w):
        out, pc = self.bufs(w)
        G.gdn_verify_step(self.cfg(G), to_dev(w["x"]), self.conv_w, self.cs, self.S, to_dev(w["alpha"]),
                          to_dev(w["beta"]), to_dev(w["z"]), self.norm_w, out, self.slot, postconv_out=pc)
        return out, pc

    def commit(self, G, w):
        views = G.make_layer_views([dict(x=to_dev(w["x"]), alpha=to_dev(w["alpha"]), beta=to_dev(w["beta"]),
                                         conv_w=self.conv_w, conv_state=self.cs, state=self.S)], "cuda")
        G.gdn_commit_layers(self.cfg(G), views, 1, self.slot, to_dev(w["n_keep"]), w["T"])

    def lazy(self, G, wp, w, dev_err=None):
        out, pc = self.bufs(w)
        G.gdn_verify_step_lazy(self.cfg(G, dev_err), to_dev(wp["x"]), to_dev(wp["alpha"]), to_dev(wp["beta"]),
                               to_dev(wp["n_keep"]), to_dev(w["x"]), self.conv_w, self.cs, self.S,
                               to_dev(w["alpha"]), to_dev(w["beta"]), to_dev(w["z"]), self.norm_w, out,
                               self.slot, postconv_out=pc)
        return out, pc


@pytest.mark.parametrize("prev_T,T,act", [(4, 4, "bf16"), (8, 3, "bf16"), (1, 8, "bf16"), (5, 2, "f32")])
def test_lazy_equals_commit_then_verify(G, orc, prev_T, T, act):
    wp, w = _windows(6, [prev_T, T], act, seed=700 + 10 * prev_T + T)
    ref, lz = Pools(wp), Pools(wp)
    ref.commit(G, wp)
    out_r, _ = ref.verify(G, w)
    out_l, pc_l = lz.lazy(G, wp, w)
    torch.cuda.synchronize()
    assert np.array_equal(bits(lz.S), bits(ref.S)), "lazy commit == gdn_commit_layers (bitwise)"
    assert np.array_equal(bits(lz.cs), bits(ref.cs))
    # the oracle: commit of the accepted prefix, then the verify from the committed pools
    cs, st = orc.commit(wp["x"], wp["alpha"], wp["beta"], wp["conv_w"], wp["conv_state"], wp["state"],
                        wp["slot_idx"], wp["n_keep"], HK, HV)
    out, pc, _, _ = orc.verify(w["x"], w["conv_w"], cs, st, w["alpha"], w["beta"], w["z"], w["norm_w"],
                               w["slot_idx"], HK, HV)
    live = [b for b in range(6) if w["slot_idx"][b] >= 0]
    if act == "bf16":
        check_bf16(to_np(out_l)[live], out[live], what=f"lazy out prev_T={prev_T} T={T}")
        check_bf16(to_np(out_l)[live], to_np(out_r)[live], what="lazy vs verify after commit")
    else:
        check_f32_out(to_np(out_l)[live], out[live], 1e-4, "lazy f32 out")
    if act == "bf16":
        check_bf16(to_np(pc_l)[live], pc[live], what="lazy post-conv")
    else:
        check_f32_out(to_np(pc_l)[live], pc[live], 1e-5, "lazy post-conv")
    assert np.all(to_np(out_l)[5] == 0), "padding entry must not be written"
    used = [int(s) for s in wp["slot_idx"] if s >= 0]
    check_states(to_np(lz.S), st, used, 1e-4, "lazy committed state")


def test_lazy_chain_of_windows(G, orc):
    """verify w0; lazy(w0 -> w1); lazy(w1 -> w2); commit w2  ==  (verify, commit) x 3,
    bitwise in the states, within tolerance in every window's outputs."""
    ws = _windows(5, [3, 8, 2], "bf16", seed=760)
    ref, lz = Pools(ws[0]), Pools(ws[0])
    outs_r = []
    for w in ws:
        outs_r.append(ref.verify(G, w)[0])
        ref.commit(G, w)
    outs_l = [lz.verify(G, ws[0])[0]]
    for wp, w in zip(ws[:-1], ws[1:]):
        outs_l.append(lz.lazy(G, wp, w)[0])
    lz.commit(G, ws[-1])
    torch.cuda.synchronize()
    assert np.array_equal(bits(lz.S), bits(ref.S)), "chained lazy windows == verify/commit (bitwise)"
    assert np.array_equal(bits(lz.cs), bits(ref.cs))
    live = [b for b in range(5) if ws[0]["slot_idx"][b] >= 0]
    for i, (a, r) in enumerate(zip(outs_l, outs_r)):
        check_bf16(to_np(a)[live], to_np(r)[live], what=f"window {i} outputs")


def test_lazy_bad_n_keep_skips_the_sequence(G):
    wp, w = _windows(4, [3, 2], "bf16", seed=790, pad=0)
    wp["n_keep"][2] = 4                                          # > prev_T
    P = Pools(wp)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _ = P.lazy(G, wp, w, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & G.GDN_DEVERR_NKEEP
    sl = int(wp["slot_idx"][2])
    assert np.array_equal(bits(P.S)[sl], wp["state"][sl].view(np.int32))
    assert np.array_equal(bits(P.cs)[sl], wp["conv_state"][sl].view(np.int16))
    assert np.all(to_np(out)[2] == 0)
