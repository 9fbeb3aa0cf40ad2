"""GPU parity of the causal conv (+SiLU, +L2 norm) and the standalone post-conv
norm against the CPU oracle, through the C ABI."""
import numpy as np
import pytest

from gated_deltanet_linear_12_gb300 import synthetic as syn
from tests.helpers import (Canary, bits, check_bf16, check_f32_cond, check_f32_rel, conv_kappa, to_dev,
                           to_np)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def G():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_linear_12_gb300 import gdn
    gdn.load()
    return gdn


def _run_conv(G, inp, fuse_norm=True, ld_pad=0, dev_err=None):
    act = torch.bfloat16 if inp["act"] == "bf16" else torch.float32
    C = inp["C"]
    x = to_dev(inp["x"])
    if ld_pad:
        xb = torch.zeros(x.shape[0], C + ld_pad, dtype=x.dtype, device="cuda")
        xb[:, :C] = x
        x = xb[:, :C]
    y = torch.zeros(inp["n_tok"], C + ld_pad, dtype=act, device="cuda")[:, :C]
    cs = to_dev(inp["conv_state"])
    cfg = G.make_config(inp["Hk"], inp["Hv"], act, cs.shape[0], dev_err=dev_err)
    G.gdn_conv_fwd(cfg, x, y, to_dev(inp["conv_w"]), cs, to_dev(inp["slot_idx"]),
                   to_dev(inp["cu_seqlens"]), to_dev(inp["has_init_conv"]), fuse_norm=fuse_norm)
    torch.cuda.synchronize()
    return y, cs


def _oracle_conv(orc, inp, fuse_norm=True, prec="f64"):
    return orc.conv_fwd(inp["x"], inp["conv_w"], inp["conv_state"], inp["slot_idx"],
                        inp["cu_seqlens"], inp["has_init_conv"], inp["Hk"], inp["Hv"],
                        l2norm=fuse_norm, prec=prec)


@pytest.mark.parametrize("fuse_norm", [True, False])
def test_conv_tiny_f32(G, orc, fuse_norm):
    """The f32 arm: against the float instantiation (same tap-ordered sum, so
    equal pre-activations; SiLU by other means) at 1e-5 relative, and against
    the double one at 1e-5 of the sum's conditioning."""
    inp = syn.workload_prefill("tiny-f32")
    y, cs = _run_conv(G, inp, fuse_norm)
    ry32, _ = _oracle_conv(orc, inp, fuse_norm, prec="f32")
    check_f32_rel(to_np(y), ry32, 1e-5, "conv f32 vs float oracle")
    ry, rcs = _oracle_conv(orc, inp, fuse_norm)
    kappa = conv_kappa(orc, inp["x"], inp["conv_w"], inp["conv_state"], inp["slot_idx"],
                       inp["cu_seqlens"], inp["has_init_conv"], inp["Hk"], inp["Hv"], l2norm=fuse_norm)
    check_f32_cond(to_np(y), ry, kappa, 1e-5, "conv f32 vs double oracle")
    assert np.array_equal(to_np(cs), rcs), "conv_state commit must be bit-exact"


@pytest.mark.parametrize("lens,init", [
    ([1, 2, 3, 63, 64, 65, 130, 200], [1, 0, 1, 0, 1, 0, 1, 1]),
    ([0, 5, 0, 129], [1, 1, 0, 1]),                   # empty sequences commit too
])
def test_conv_varlen_bf16(G, orc, lens, init):
    inp = syn.prefill_inputs(lens, 2, 4, "bf16", seed=101, init_mask=np.array(init))
    guard = Canary()
    act = torch.bfloat16
    y = guard.wrap(torch.zeros(inp["n_tok"], inp["C"], dtype=act, device="cuda"))
    cs = guard.wrap(to_dev(inp["conv_state"]))
    cfg = G.make_config(inp["Hk"], inp["Hv"], act, cs.shape[0])
    G.gdn_conv_fwd(cfg, guard.wrap(to_dev(inp["x"])), y, to_dev(inp["conv_w"]), cs,
                   to_dev(inp["slot_idx"]), to_dev(inp["cu_seqlens"]), to_dev(inp["has_init_conv"]))
    torch.cuda.synchronize()
    guard.check("conv")
    ry, rcs = _oracle_conv(orc, inp)
    check_bf16(to_np(y), ry, what="conv bf16")
    assert np.array_equal(to_np(cs), rcs), "conv_state commit must be bit-exact"


def test_conv_many_sequences_bf16(G, orc):
    """40 sequences (more than one 32-lane group of the chunk lookup), with empty
    and 1..5-token ones among them: outputs against the oracle, conv_state rows
    of every slot bit-exact."""
    rng = np.random.default_rng(107)
    lens = rng.integers(0, 140, size=40)
    lens[[3, 17, 31]] = 0
    lens[[5, 6, 7, 8, 9]] = [1, 2, 3, 4, 5]
    init = rng.integers(0, 2, size=40).astype(np.uint8)
    inp = syn.prefill_inputs(lens, 2, 4, "bf16", seed=107, init_mask=init)
    y, cs = _run_conv(G, inp)
    ry, rcs = _oracle_conv(orc, inp)
    check_bf16(to_np(y), ry, what="conv bf16, 40 sequences")
    assert np.array_equal(to_np(cs), rcs), "conv_state commit must be bit-exact"


@pytest.mark.parametrize("act", ["bf16", "f32"])
def test_conv_tail_group_of_one_head(G, orc, act):
    """Hk = 1, Hv = 3: 5 heads, so the last group of four holds one head and half
    of each warp's lanes are idle (they still take part in the norm's lane
    exchanges); outputs against the oracle, conv_state bit-exact."""
    inp = syn.prefill_inputs([70, 1, 0, 129], 1, 3, act, seed=108, init_mask=np.array([1, 0, 1, 1]))
    y, cs = _run_conv(G, inp)
    ry, rcs = _oracle_conv(orc, inp)
    if act == "bf16":
        check_bf16(to_np(y), ry, what="conv bf16, 5 heads")
    else:
        ry32, _ = _oracle_conv(orc, inp, prec="f32")
        check_f32_rel(to_np(y), ry32, 1e-5, "conv f32, 5 heads")
    assert np.array_equal(to_np(cs), rcs), "conv_state commit must be bit-exact"


def test_conv_padded_rows_and_padding_sequence(G, orc):
    inp = syn.prefill_inputs([70, 9, 33], 1, 2, "bf16", seed=102, init_mask=np.array([1, 1, 0]))
    inp["slot_idx"][1] = -1
    y, cs = _run_conv(G, inp, ld_pad=64)
    ry, rcs = _oracle_conv(orc, inp)
    yy = to_np(y)
    check_bf16(yy, ry, what="conv ld>C")
    assert np.all(yy[70:79] == 0), "padding sequence rows must stay untouched"
    assert np.array_equal(to_np(cs), rcs)


def test_fused_norm_equals_conv_then_postconv_norm_bitwise(G):
    inp = syn.prefill_inputs([100, 37], 2, 4, "f32", seed=103, init_mask=np.array([1, 0]))
    y_fused, _ = _run_conv(G, inp, fuse_norm=True)
    y_plain, _ = _run_conv(G, inp, fuse_norm=False)
    cfg = G.make_config(2, 4, torch.float32, inp["conv_state"].shape[0])
    y2 = torch.empty_like(y_plain)
    G.gdn_postconv_norm(cfg, y_plain, y2)
    torch.cuda.synchronize()
    assert np.array_equal(bits(y2), bits(y_fused))


def test_postconv_norm_f32_bitwise(G, orc):
    """The f32 arm: any change of the reduction order shows up here."""
    Hk, Hv = 1, 3
    rows = syn.random_f32_rows(3000, syn.channels(Hk, Hv), seed=104, scale=2.0)
    cfg = G.make_config(Hk, Hv, torch.float32, 1)
    yi = to_dev(rows)
    yo = torch.empty_like(yi)
    G.gdn_postconv_norm(cfg, yi, yo)
    torch.cuda.synchronize()
    ref = orc.l2norm(rows, Hk, Hv, prec="f32")
    assert np.array_equal(bits(yo), ref.astype(np.float32).view(np.int32))
    # in place gives the same bits
    G.gdn_postconv_norm(cfg, yi, yi)
    torch.cuda.synchronize()
    assert np.array_equal(bits(yi), bits(yo))


@pytest.mark.parametrize("in_t,out_t", [("f32", "bf16"), ("bf16", "bf16"), ("bf16", "f32")])
def test_postconv_norm_mixed_types(G, orc, in_t, out_t):
    Hk, Hv = 2, 4
    rows = syn.random_f32_rows(500, syn.channels(Hk, Hv), seed=105)
    src = syn.to_act(rows, in_t)
    yi = to_dev(src)
    yo = torch.empty(rows.shape, dtype=torch.bfloat16 if out_t == "bf16" else torch.float32,
                     device="cuda")
    cfg = G.make_config(Hk, Hv, torch.bfloat16, 1)
    G.gdn_postconv_norm(cfg, yi, yo)
    torch.cuda.synchronize()
    ref = orc.l2norm(src, Hk, Hv, prec="f32")
    if out_t == "bf16":
        check_bf16(to_np(yo), ref, what="postconv bf16")
    else:
        assert np.array_equal(bits(yo), ref.astype(np.float32).view(np.int32))


def test_conv_bad_slot_sets_error_bit(G, orc):
    inp = syn.prefill_inputs([10, 20], 1, 1, "bf16", seed=106, init_mask=np.array([1, 1]))
    n_slots = inp["conv_state"].shape[0]
    inp["slot_idx"][0] = n_slots + 5
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y, cs = _run_conv(G, inp, dev_err=err)
    assert int(err.item()) & G.GDN_DEVERR_SLOT
    assert np.all(to_np(y)[:10] == 0)
    ry, rcs = _oracle_conv(orc, dict(inp, slot_idx=np.array([-1, inp["slot_idx"][1]], np.int32)))
    check_bf16(to_np(y)[10:], ry[10:], what="valid sequence")
    assert np.array_equal(to_np(cs), rcs)


@pytest.mark.slow
def test_conv_full_varlen_prefill_workload(G, orc):
    """The varlen-prefill workload at full size; sampled heads checked by the oracle."""
    inp = syn.workload_prefill("varlen-prefill-bf16")
    y, cs = _run_conv(G, inp)
    yy = to_np(y)
    # full-channel oracle on a few sequences
    for s in (0, 3, 7):
        t0, t1 = inp["cu_seqlens"][s], inp["cu_seqlens"][s + 1]
        sub = dict(inp, x=inp["x"][t0:t1], cu_seqlens=np.array([0, t1 - t0], np.int32),
                   slot_idx=inp["slot_idx"][s:s + 1], has_init_conv=inp["has_init_conv"][s:s + 1])
        ry, rcs = _oracle_conv(orc, sub)
        check_bf16(yy[t0:t1], ry, what=f"seq {s}")
        slot = inp["slot_idx"][s]
        assert np.array_equal(to_np(cs)[slot], rcs[slot])
