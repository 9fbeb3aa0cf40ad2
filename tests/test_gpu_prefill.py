"""GPU parity of the chunked prefill (conv -> delta rule -> gated RMSNorm)
against the CPU oracle, through the C ABI."""
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


def _oracle_qkv(orc, inp):
    """Post-conv activations as stored: the double oracle's values rounded to
    the activation dtype (to nearest even for bf16, to f32 otherwise)."""
    y, _ = orc.conv_fwd(inp["x"], inp["conv_w"], inp["conv_state"], inp["slot_idx"],
                        inp["cu_seqlens"], inp["has_init_conv"], inp["Hk"], inp["Hv"])
    if inp["act"] == "bf16":
        y = orc.round_bf16(y)
    return syn.to_act(y.astype(np.float32), inp["act"])


def _run_prefill(G, inp, qkv, dev_err=None, q_scale=1.0, eps=1e-6):
    """The prefill with its outputs and state pool between NaN guard bands."""
    act = torch.bfloat16 if inp["act"] == "bf16" else torch.float32
    guard = Canary()
    S = guard.wrap(to_dev(inp["state"]))
    out = guard.wrap(torch.zeros(inp["n_tok"], inp["Hv"] * 128, dtype=act, device="cuda"))
    cfg = G.make_config(inp["Hk"], inp["Hv"], act, S.shape[0], dev_err=dev_err, q_scale=q_scale, eps=eps)
    G.gdn_delta_prefill(cfg, guard.wrap(to_dev(qkv)), to_dev(inp["alpha"]), to_dev(inp["beta"]),
                        guard.wrap(to_dev(inp["z"])), to_dev(inp["norm_w"]), out, S,
                        to_dev(inp["slot_idx"]), to_dev(inp["cu_seqlens"]), to_dev(inp["has_init_state"]))
    torch.cuda.synchronize()
    guard.check("prefill")
    return out, S


def _oracle_prefill(orc, inp, qkv, q_scale=1.0, eps=1e-6):
    return orc.prefill(qkv, inp["alpha"], inp["beta"], inp["z"], inp["norm_w"], inp["state"],
                       inp["slot_idx"], inp["cu_seqlens"], inp["has_init_state"], inp["Hk"],
                       inp["Hv"], q_scale=q_scale, eps=eps)


def test_prefill_tiny_f32(G, orc):
    inp = syn.workload_prefill("tiny-f32")
    qkv = _oracle_qkv(orc, inp)
    out, S = _run_prefill(G, inp, qkv)
    ro, rs = _oracle_prefill(orc, inp, qkv)
    check_f32_out(to_np(out), ro, 1e-4, "prefill f32 out")
    check_states(to_np(S), rs, [int(inp["slot_idx"][0])], 1e-4, "prefill f32 state")


@pytest.mark.parametrize("lens,init", [
    ([1, 63, 64, 65, 200, 3], [1, 0, 1, 1, 0, 1]),
    ([0, 130, 0], [1, 1, 0]),
])
def test_prefill_varlen_bf16(G, orc, lens, init):
    inp = syn.prefill_inputs(lens, 2, 4, "bf16", seed=500 + len(lens), init_mask=np.array(init))
    qkv = _oracle_qkv(orc, inp)
    out, S = _run_prefill(G, inp, qkv)
    ro, rs = _oracle_prefill(orc, inp, qkv)
    check_bf16(to_np(out), ro, what="prefill bf16 out")
    check_states(to_np(S), rs, [int(s) for s in inp["slot_idx"]], 1e-4, "prefill bf16 state")
    unused = sorted(set(range(inp["state"].shape[0])) - set(int(s) for s in inp["slot_idx"]))
    for sl in unused:
        assert np.array_equal(bits(S)[sl], inp["state"][sl].view(np.int32))


def test_prefill_many_sequences_bf16(G, orc):
    """300 sequences (past the 256 the block ranking by length covers; the blocks
    then take sequences in index order), lengths 0..100: outputs and every state
    against the oracle, untouched slots bitwise unchanged."""
    rng = np.random.default_rng(570)
    lens = rng.integers(0, 101, size=300)
    lens[[0, 150, 299]] = 0
    init = rng.integers(0, 2, size=300).astype(np.uint8)
    inp = syn.prefill_inputs(lens, 1, 2, "bf16", seed=570, init_mask=init)
    qkv = _oracle_qkv(orc, inp)
    out, S = _run_prefill(G, inp, qkv)
    ro, rs = _oracle_prefill(orc, inp, qkv)
    check_bf16(to_np(out), ro, what="prefill bf16 out, 300 sequences")
    check_states(to_np(S), rs, [int(s) for s in inp["slot_idx"]], 1e-4, "prefill bf16 state, 300 sequences")
    unused = sorted(set(range(inp["state"].shape[0])) - set(int(s) for s in inp["slot_idx"]))
    for sl in unused:
        assert np.array_equal(bits(S)[sl], inp["state"][sl].view(np.int32))


@pytest.mark.parametrize("act", ["bf16", "f32"])
def test_prefill_q_scale_and_eps(G, orc, act):
    """q_scale = d^-1/2 (an ABI parameter the definition does not have) with an eps
    large enough that the output RMSNorm does not divide the scale away."""
    inp = syn.prefill_inputs([70, 129], 2, 4, act, seed=530, init_mask=np.array([1, 0]))
    qkv = _oracle_qkv(orc, inp)
    qs, eps = 128 ** -0.5, 0.05
    out, S = _run_prefill(G, inp, qkv, q_scale=qs, eps=eps)
    ro, rs = _oracle_prefill(orc, inp, qkv, q_scale=qs, eps=eps)
    if act == "bf16":
        check_bf16(to_np(out), ro, what="prefill q_scale out")
    else:
        check_f32_out(to_np(out), ro, 1e-4, "prefill q_scale out")
    check_states(to_np(S), rs, [int(s) for s in inp["slot_idx"]], 1e-4, "prefill q_scale state")


@pytest.mark.parametrize("lens,init", [([1, 63, 64, 65, 200, 3], [1, 0, 1, 1, 0, 1]), ([300, 17], [0, 1])])
def test_prefill_tc_f32_out(G, orc, lens, init):
    """The f32-output arm of the tensor-core prefill (bf16 activations): the
    outputs before any rounding against the f32 recurrence tolerance."""
    inp = syn.prefill_inputs(lens, 2, 4, "bf16", seed=560 + len(lens), init_mask=np.array(init),
                             gate_form="softplus")
    qkv = _oracle_qkv(orc, inp)
    S = to_dev(inp["state"])
    out = torch.zeros(inp["n_tok"], inp["Hv"] * 128, dtype=torch.float32, device="cuda")
    cfg = G.make_config(inp["Hk"], inp["Hv"], torch.bfloat16, S.shape[0], out_f32=True)
    G.gdn_delta_prefill(cfg, to_dev(qkv), to_dev(inp["alpha"]), to_dev(inp["beta"]), to_dev(inp["z"]),
                        to_dev(inp["norm_w"]), out, S, to_dev(inp["slot_idx"]), to_dev(inp["cu_seqlens"]),
                        to_dev(inp["has_init_state"]))
    torch.cuda.synchronize()
    ro, rs = _oracle_prefill(orc, inp, qkv)
    check_f32_out(to_np(out), ro, 1e-4, "prefill tc f32 out")
    check_states(to_np(S), rs, [int(s) for s in inp["slot_idx"]], 1e-4, "prefill tc f32-out state")


def test_prefill_group_of_three(G, orc):
    inp = syn.prefill_inputs([90, 17], 2, 6, "bf16", seed=520, init_mask=np.array([1, 0]))
    qkv = _oracle_qkv(orc, inp)
    out, S = _run_prefill(G, inp, qkv)
    ro, rs = _oracle_prefill(orc, inp, qkv)
    check_bf16(to_np(out), ro, what="prefill G=3")
    check_states(to_np(S), rs, [int(s) for s in inp["slot_idx"]], 1e-4, "prefill G=3 state")


def test_conv_then_prefill_end_to_end(G, orc):
    """Both GPU entry points chained, against the oracle's own chain."""
    inp = syn.prefill_inputs([150, 70], 2, 4, "bf16", seed=530, init_mask=np.array([1, 1]))
    act = torch.bfloat16
    x = to_dev(inp["x"])
    y = torch.empty_like(x)
    cs = to_dev(inp["conv_state"])
    cfg = G.make_config(2, 4, act, cs.shape[0])
    G.gdn_conv_fwd(cfg, x, y, to_dev(inp["conv_w"]), cs, to_dev(inp["slot_idx"]),
                   to_dev(inp["cu_seqlens"]), to_dev(inp["has_init_conv"]))
    S = to_dev(inp["state"])
    out = torch.zeros(inp["n_tok"], 4 * 128, dtype=act, device="cuda")
    G.gdn_delta_prefill(cfg, y, to_dev(inp["alpha"]), to_dev(inp["beta"]), to_dev(inp["z"]),
                        to_dev(inp["norm_w"]), out, S, to_dev(inp["slot_idx"]),
                        to_dev(inp["cu_seqlens"]), to_dev(inp["has_init_state"]))
    torch.cuda.synchronize()
    y64, _ = orc.conv_fwd(inp["x"], inp["conv_w"], inp["conv_state"], inp["slot_idx"],
                          inp["cu_seqlens"], inp["has_init_conv"], 2, 4)
    check_bf16(to_np(y), y64, what="chain post-conv")
    qkv = _oracle_qkv(orc, inp)
    ro, rs = _oracle_prefill(orc, inp, qkv)
    check_bf16(to_np(out), ro, what="chain out")
    check_states(to_np(S), rs, [int(s) for s in inp["slot_idx"]], 1e-4, "chain state")


def test_prefill_then_verify_equals_longer_prefill(G, orc):
    """Phase composition on the GPU: prefill(n) then a verify of the next T
    tokens from the committed pools, against the oracle's prefill(n) then
    verify(T). The oracle pins (P8) show that chain equals one prefill of n + T
    tokens when the activations are rounded alike; here the verify keeps them
    unrounded, as the fused kernel does."""
    n, T = 100, 5
    inp = syn.prefill_inputs([n + T], 2, 4, "bf16", seed=540, init_mask=np.array([1]),
                             slot_perm=False, n_slots=1)
    act = torch.bfloat16
    C = inp["C"]
    cfg = G.make_config(2, 4, act, 1)
    x = to_dev(inp["x"])
    cs = to_dev(inp["conv_state"])
    S = to_dev(inp["state"])
    cw = to_dev(inp["conv_w"])
    y = torch.empty(n, C, dtype=act, device="cuda")
    one = torch.ones(1, dtype=torch.uint8, device="cuda")
    slot = torch.zeros(1, dtype=torch.int32, device="cuda")
    cu = torch.tensor([0, n], dtype=torch.int32, device="cuda")
    G.gdn_conv_fwd(cfg, x[:n], y, cw, cs, slot, cu, one)
    out_p = torch.empty(n, 512, dtype=act, device="cuda")
    al, be, z = to_dev(inp["alpha"]), to_dev(inp["beta"]), to_dev(inp["z"])
    nw = to_dev(inp["norm_w"])
    G.gdn_delta_prefill(cfg, y, al[:n].contiguous(), be[:n].contiguous(), z[:n].contiguous(), nw,
                        out_p, S, slot, cu, one)
    out_v = torch.empty(1, T, 512, dtype=act, device="cuda")
    G.gdn_verify_step(cfg, x[n:].reshape(1, T, C).contiguous(), cw, cs, S,
                      al[n:].reshape(1, T, 4).contiguous(), be[n:].reshape(1, T, 4).contiguous(),
                      z[n:].reshape(1, T, 512).contiguous(), nw, out_v, slot)
    torch.cuda.synchronize()
    qkv = _oracle_qkv(orc, inp)
    ro, _ = _oracle_prefill(orc, inp, qkv)
    check_bf16(to_np(out_p), ro[:n], what="prefill part")
    # the oracle's chain: prefill of the first n tokens, then the verify
    sub = dict(inp, x=inp["x"][:n], alpha=inp["alpha"][:n], beta=inp["beta"][:n], z=inp["z"][:n],
               cu_seqlens=np.array([0, n], np.int32), n_tok=n)
    _, cs1 = orc.conv_fwd(sub["x"], inp["conv_w"], inp["conv_state"], [0], sub["cu_seqlens"], [1], 2, 4)
    _, st1 = _oracle_prefill(orc, sub, qkv[:n])
    rv, _, _, _ = orc.verify(inp["x"][None, n:], inp["conv_w"], cs1, st1, inp["alpha"][None, n:],
                             inp["beta"][None, n:], inp["z"][None, n:], inp["norm_w"], [0], 2, 4)
    check_bf16(to_np(out_v), rv, what="verify after prefill")
