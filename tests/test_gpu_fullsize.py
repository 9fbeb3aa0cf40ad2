"""Parity at the full workload sizes, in the launch configurations bench.py
times. The GPU runs the whole workload; the oracle checks sampled (sequence,
head) chains built from channel slices (heads are independent), or everything
where that is cheap (verify window, decode layer)."""
import numpy as np
import pytest

from gated_deltanet_linear_12_gb300 import synthetic as syn
from tests.helpers import bits, check_bf16, check_states, to_dev, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
D = 128


@pytest.fixture(scope="module")
def G():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_linear_12_gb300 import gdn
    gdn.load()
    return gdn


def _gpu_prefill_chain(G, inp):
    act = torch.bfloat16
    x = to_dev(inp["x"])
    y = torch.empty_like(x)
    cs = to_dev(inp["conv_state"])
    S = to_dev(inp["state"])
    cfg = G.make_config(inp["Hk"], inp["Hv"], act, S.shape[0])
    slot, cu = to_dev(inp["slot_idx"]), to_dev(inp["cu_seqlens"])
    G.gdn_conv_fwd(cfg, x, y, to_dev(inp["conv_w"]), cs, slot, cu, to_dev(inp["has_init_conv"]))
    out = torch.empty(inp["n_tok"], inp["Hv"] * D, dtype=act, device="cuda")
    G.gdn_delta_prefill(cfg, y, to_dev(inp["alpha"]), to_dev(inp["beta"]), to_dev(inp["z"]),
                        to_dev(inp["norm_w"]), out, S, slot, cu, to_dev(inp["has_init_state"]))
    torch.cuda.synchronize()
    return y, out, S, cs


def _oracle_chain(orc, inp, s, h):
    """Oracle conv + prefill of sequence s, v head h, on its own channels: the
    double conv (returned unrounded), rounded to bf16 as stored rows, then the
    token-by-token recurrence."""
    Hk, Hv = inp["Hk"], inp["Hv"]
    hq = h // (Hv // Hk)
    chans = np.r_[hq * D:(hq + 1) * D, (Hk + hq) * D:(Hk + hq + 1) * D,
                  (2 * Hk + h) * D:(2 * Hk + h + 1) * D]
    t0, t1 = int(inp["cu_seqlens"][s]), int(inp["cu_seqlens"][s + 1])
    slot = int(inp["slot_idx"][s])
    x = inp["x"][t0:t1][:, chans]
    cu = np.array([0, t1 - t0], np.int32)
    y, _ = orc.conv_fwd(x, inp["conv_w"][chans], inp["conv_state"][slot:slot + 1][:, :, chans], [0],
                        cu, inp["has_init_conv"][s:s + 1], 1, 1)
    qkv = syn.to_act(orc.round_bf16(y).astype(np.float32), "bf16")
    hd = slice(h * D, (h + 1) * D)
    out, st = orc.prefill(qkv, inp["alpha"][t0:t1, h:h + 1], inp["beta"][t0:t1, h:h + 1],
                          inp["z"][t0:t1, hd], inp["norm_w"], inp["state"][slot:slot + 1, h:h + 1],
                          [0], cu, inp["has_init_state"][s:s + 1], 1, 1)
    return y, out, st[0, 0], (t0, t1, slot, chans)


@pytest.mark.parametrize("name,samples", [
    ("varlen-prefill-bf16", [(1, 0), (1, 31), (4, 7), (3, 16)]),
    ("long-prefill-bf16", [(0, 0), (3, 29)]),
])
def test_prefill_workload_full_size(G, orc, name, samples):
    inp = syn.workload_prefill(name)
    y, out, S, cs = _gpu_prefill_chain(G, inp)
    for s, h in samples:
        y64, ro, rs, (t0, t1, slot, chans) = _oracle_chain(orc, inp, s, h)
        ci = torch.as_tensor(chans, device="cuda")
        check_bf16(to_np(y[t0:t1].index_select(1, ci)), y64, what=f"{name} post-conv seq {s}")
        check_bf16(to_np(out[t0:t1, h * D:(h + 1) * D]), ro, what=f"{name} seq {s} head {h}")
        check_states(to_np(S[slot:slot + 1, h:h + 1]), rs[None, None], [0], 1e-4, f"{name} state")


def test_spec_verify_window_full_size(G, orc):
    """B = 32, T = 8, C = 8192: verify of every sequence and a 3-layer batched
    commit, each checked in full against the oracle."""
    B, T, L = 32, 8, 3
    inps = [syn.verify_inputs(B, T, 16, 32, "bf16", seed=syn.seed_of("spec-verify-bf16") + l)
            for l in range(L)]
    n_keep = inps[0]["n_keep"]
    bf = torch.bfloat16
    layers = []
    for inp in inps:
        inp["n_keep"] = n_keep
        inp["slot_idx"] = inps[0]["slot_idx"]
        d = dict(x=to_dev(inp["x"]), conv_w=to_dev(inp["conv_w"]), conv_state=to_dev(inp["conv_state"]),
                 state=to_dev(inp["state"]), alpha=to_dev(inp["alpha"]), beta=to_dev(inp["beta"]))
        layers.append(d)
    cfg = G.make_config(16, 32, bf, inps[0]["state"].shape[0])
    slot = to_dev(inps[0]["slot_idx"])
    outs = []
    for inp, lay in zip(inps, layers):
        out = torch.empty(B, T, 32 * D, dtype=bf, device="cuda")
        G.gdn_verify_step(cfg, lay["x"], lay["conv_w"], lay["conv_state"], lay["state"], lay["alpha"],
                          lay["beta"], to_dev(inp["z"]), to_dev(inp["norm_w"]), out, slot)
        outs.append(out)
    views = G.make_layer_views(layers, "cuda")
    G.gdn_commit_layers(cfg, views, L, slot, to_dev(n_keep), T)
    torch.cuda.synchronize()
    for l, inp in enumerate(inps):
        ro, _, _, _ = orc.verify(inp["x"], inp["conv_w"], inp["conv_state"], inp["state"],
                                 inp["alpha"], inp["beta"], inp["z"], inp["norm_w"], inp["slot_idx"],
                                 16, 32)
        check_bf16(to_np(outs[l]), ro, what=f"layer {l} verify")
        rcs, rst = orc.commit(inp["x"], inp["alpha"], inp["beta"], inp["conv_w"], inp["conv_state"],
                              inp["state"], inp["slot_idx"], n_keep, 16, 32)
        assert np.array_equal(to_np(layers[l]["conv_state"]), rcs), "conv_state commit bit-exact"
        check_states(to_np(layers[l]["state"]), rst, range(rst.shape[0]), 1e-4, f"layer {l} commit")


def test_decode_layer_full_size(G, orc):
    """B = 256, T = 1, every token accepted, one full layer."""
    B = 256
    inp = syn.verify_inputs(B, 1, 16, 32, "bf16", seed=syn.seed_of("decode-bf16"))
    bf = torch.bfloat16
    cs, S = to_dev(inp["conv_state"]), to_dev(inp["state"])
    cfg = G.make_config(16, 32, bf, S.shape[0])
    out = torch.empty(B, 1, 32 * D, dtype=bf, device="cuda")
    G.gdn_verify_step(cfg, to_dev(inp["x"]), to_dev(inp["conv_w"]), cs, S, to_dev(inp["alpha"]),
                      to_dev(inp["beta"]), to_dev(inp["z"]), to_dev(inp["norm_w"]), out,
                      to_dev(inp["slot_idx"]), commit_all=True)
    torch.cuda.synchronize()
    ro, _, rcs, rst = orc.verify(inp["x"], inp["conv_w"], inp["conv_state"], inp["state"],
                                 inp["alpha"], inp["beta"], inp["z"], inp["norm_w"], inp["slot_idx"],
                                 16, 32, commit_all=True)
    check_bf16(to_np(out), ro, what="decode outputs")
    assert np.array_equal(to_np(cs), rcs), "conv_state commit bit-exact"
    check_states(to_np(S), rst, range(rst.shape[0]), 1e-4, "decode state")
