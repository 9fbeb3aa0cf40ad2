"""The bench's roofline choice for the prefill on the CPU: the binding roofline is
the one with the longer floor (algorithmic bytes at the HBM peak, or algorithmic
FLOPs at the peak of the unit the products run on)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

bench = pytest.importorskip("bench")

PEAKS = {"hbm_gbs": 6684.5, "bf16_tflops": 1882.8, "sm_max_mhz": 2070.0}

# varlen prefill workload: 6157 tokens, 8 sequences (6 with an initial state), C = 8192, Hv = 32
N_TOK, C, HV = 6157, 8192, 32


def test_bf16_prefill_is_bound_by_hbm():
    """155 FLOP per byte is below the bf16 ridge of 1882.8 / 6684.5 * 1e3 = 282 FLOP per
    byte, so the bytes' floor is the longer one."""
    flops = bench.prefill_delta_flops(N_TOK, HV)
    nbytes = bench.prefill_delta_bytes(N_TOK, C, HV, 6, 8)
    assert 150 < flops / nbytes < 160
    r = bench.prefill_roofline("prefill_tc_kernel", flops, nbytes, 0.316, PEAKS, "measured", 123)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == PEAKS["hbm_gbs"]
    assert r["floor_us"]["hbm"] > r["floor_us"]["tensor"]
    assert r["achieved"] == pytest.approx(nbytes / 0.316e-3 / 1e9, rel=1e-3)
    assert r["frac"] == pytest.approx(r["achieved"] / PEAKS["hbm_gbs"], rel=1e-3)
    assert r["tensor_frac"] == pytest.approx(flops / 0.316e-3 / 1e12 / PEAKS["bf16_tflops"], rel=1e-3)
    assert r["traffic"] == 123


def test_f32_prefill_is_bound_by_the_fp32_pipe():
    flops = bench.prefill_delta_flops(N_TOK, HV)
    nbytes = bench.prefill_delta_bytes(N_TOK, C, HV, 6, 8, es=4)
    r = bench.prefill_roofline("prefill_ffma_kernel", flops, nbytes, 2.0, PEAKS, "measured", 123)
    assert r["bound"] == "alu" and r["unit"] == "TFLOP/s"
    assert r["peak"] == pytest.approx(152 * 128 * 2 * 2070e6 / 1e12, rel=1e-3)
    assert r["floor_us"]["alu"] > r["floor_us"]["hbm"]
    assert r["traffic"] is None


def test_a_compute_heavy_launch_is_bound_by_the_tensor_pipe():
    r = bench.prefill_roofline("prefill_tc_kernel", 1e12, 1e6, 1.0, PEAKS, "measured", None)
    assert r["bound"] == "tensor" and r["frac"] == pytest.approx(1.0 / PEAKS["bf16_tflops"] * 1e3, rel=1e-3)
