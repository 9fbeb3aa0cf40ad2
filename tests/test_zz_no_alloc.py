"""The allocation-free verify entry point (gdn_verify_step_noalloc), for callers
that cannot allocate device memory themselves (code hosted in a runtime that
owns every device allocation, services on a fixed memory budget, loops that
must not synchronise through cudaMalloc). It is the read-only verify with no
workspace; it launches the same kernel as gdn_verify_step. Checked against
gdn_verify_step on two calls in a row of different shapes, and the device's
free memory around a pair of calls on two streams. This file is collected
last."""
import ctypes

import numpy as np
import pytest

from gated_deltanet_linear_12_gb300 import synthetic as syn
from tests.helpers import bits, check_bf16, to_dev, to_np

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


def _verify_both(G, inp):
    act = torch.bfloat16
    d = {k: to_dev(inp[k]) for k in ("x", "conv_w", "conv_state", "state", "alpha", "beta", "z",
                                      "norm_w", "slot_idx")}
    cfg = G.make_config(inp["Hk"], inp["Hv"], act, d["state"].shape[0])
    B, T, Hv = inp["B"], inp["T"], inp["Hv"]
    ref = torch.zeros(B, T, Hv * D, dtype=act, device="cuda")         # padding rows stay 0
    new = torch.zeros_like(ref)
    G.gdn_verify_step(cfg, d["x"], d["conv_w"], d["conv_state"], d["state"], d["alpha"], d["beta"],
                      d["z"], d["norm_w"], ref, d["slot_idx"])
    G.gdn_verify_step_noalloc(cfg, d["x"], d["conv_w"], d["conv_state"], d["state"], d["alpha"],
                              d["beta"], d["z"], d["norm_w"], new, d["slot_idx"])
    torch.cuda.synchronize()
    # read-only: the pools are unchanged
    assert np.array_equal(bits(d["state"]), inp["state"].view(np.int32))
    return to_np(ref), to_np(new)


def test_noalloc_matches_workspace_verify_two_calls(G):
    # 1: the spec-verify window; 2: a smaller one with padding
    first = syn.verify_inputs(32, 8, 16, 32, "bf16", seed=syn.seed_of("spec-verify-bf16"))
    second = syn.verify_inputs(5, 3, 2, 4, "bf16", seed=901, pad_slots=1)
    for inp in (first, second):
        ref, new = _verify_both(G, inp)
        check_bf16(new, ref, what=f"no-alloc verify B={inp['B']} T={inp['T']}")


def test_noalloc_leaves_free_memory_unchanged(G):
    """Two calls on two streams, free device memory read before and after."""
    inp = syn.verify_inputs(8, 5, 2, 4, "bf16", seed=902)
    d = {k: to_dev(inp[k]) for k in ("x", "conv_w", "conv_state", "state", "alpha", "beta", "z",
                                      "norm_w", "slot_idx")}
    cfg = G.make_config(2, 4, torch.bfloat16, d["state"].shape[0])
    outs = [torch.zeros(8, 5, 4 * D, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    G.gdn_verify_step_noalloc(cfg, d["x"], d["conv_w"], d["conv_state"], d["state"], d["alpha"],
                              d["beta"], d["z"], d["norm_w"], outs[0], d["slot_idx"])   # warm-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for o, st in zip(outs, streams):
        G.gdn_verify_step_noalloc(cfg, d["x"], d["conv_w"], d["conv_state"], d["state"], d["alpha"],
                                  d["beta"], d["z"], d["norm_w"], o, d["slot_idx"], stream=st)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
    assert np.array_equal(bits(outs[0]), bits(outs[1]))


def test_noalloc_needs_no_memory_of_its_own(G):
    cfg = G.make_config(16, 32, torch.bfloat16, 64)
    assert G.gdn_verify_workspace_bytes(cfg, 64, 8) == 0
    lib = G.load()
    ptrs = [ctypes.c_void_p(0x7f0000000000 + i * 0x10000000) for i in range(10)]
    assert lib.gdn_verify_step_noalloc(ctypes.byref(cfg), *ptrs, 64, 9, None, None) == G.GDN_ERR_INVALID
