"""The bench's roofline choice for the prefill on the CPU: the binding roofline is
the one with the longer floor (algorithmic bytes at the HBM peak, or algorithmic
FLOPs at the peak of the unit the products run on); and its byte accounting per
unit of work (token, sequence, layer) for the prefill, verify, commit and decode."""
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


# ---------------------------------------------------------------- per-unit byte accounting
MB = 1e6


def test_verify_window_bytes_per_layer():
    """B = 32 sequences of T = 8 drafts, C = 8192, Hv = 32: the 64 MiB state read,
    x (T x 512 KiB), z and out (T x 256 KiB each), the 1.5 MiB of conv_state rows,
    about 77 MB a layer; the lazy window adds the write-back and the accepted rows."""
    v = bench.window_bytes(32, 8, 32, 8192, 1, [0] * 32)
    parts = 64 * 2**20 + 8 * 512 * 1024 + 2 * 8 * 256 * 1024 + 1.5 * 2**20
    assert abs(v["verify"] - parts) < 0.2 * MB and round(v["verify"] / MB) == 77
    assert v["commit"] == 0                                  # nothing accepted
    nk = [0, 8] + [3] * 30
    full = bench.window_bytes(32, 8, 32, 8192, 36, nk)
    lazy = bench.window_bytes(32, 8, 32, 8192, 36, nk, lazy=True)
    assert full["verify"] == 36 * v["verify"]
    per_seq_state = 32 * 128 * 128 * 4
    # a commit reads and writes S; lazy reads it once for both: one S read saved per
    # accepting sequence and layer (and a conv_state read, and conv_w per sequence)
    saved = full["verify"] + full["commit"] - lazy["verify"]
    assert saved == 36 * 31 * (per_seq_state + 3 * 8192 * 2 + 8192 * 4 * 2)


def test_decode_bytes_per_layer():
    """B = 256, T = 1: S read and written (1 GiB), conv_state rows read and written
    (24 MiB), x, z and out (8 MiB): about 1.107 GB a layer."""
    v = bench.window_bytes(256, 1, 32, 8192, 1, [1] * 256, decode=True)
    assert round(v["verify"] / 1e9, 3) == 1.107 and v["commit"] == 0


def test_prefill_bytes_per_unit():
    """Conv: 4 C bytes a token, 96 KiB of conv_state per sequence with an initial
    state (read and write), 64 KiB of weights; delta rule: 33,024 bytes a token and
    2 MiB of state per read or write."""
    C = 8192
    assert bench.prefill_conv_bytes(1, C, 0, 0) - bench.prefill_conv_bytes(0, C, 0, 0) == 4 * C
    assert bench.prefill_conv_bytes(0, C, 1, 1) - bench.prefill_conv_bytes(0, C, 0, 0) == 96 * 1024
    assert bench.prefill_conv_bytes(0, C, 0, 0) == 64 * 1024
    assert bench.prefill_delta_bytes(1, C, 32, 0, 0) == 33024
    assert bench.prefill_delta_bytes(0, C, 32, 1, 0) == 2 * 2**20
