"""Values the pages print, kept as text fixtures under tests/golden/ (each file
names its page and section), against the library's layout arithmetic."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
GOLDEN = os.path.join(ROOT, "tests", "golden")

from gated_deltanet_linear_12_gb300 import synthetic as syn  # noqa: E402


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = (s.strip() for s in line.split("="))
                vals[k] = float(v) if "." in v else int(v)
    return vals


def test_strata_verify_window_geometry():
    """"Strata PR #3226", "Benchmark Evidence": 16 q/k heads and 48 v heads of 128
    give 10240 packed channels and a value dimension of 6144, at most 8 draft
    tokens, and 117.7 MB of state over 36 layers: 48 x 128 x 128 f32 recurrent
    state plus 3 conv_state rows of 10240 channels at 4 bytes, per layer."""
    bench = pytest.importorskip("bench")
    g = _golden("strata_pr3226_geometry.txt")
    assert syn.channels(g["qk_heads"], g["v_heads"]) == g["channels"]      # [q | k | v] packing
    assert g["v_heads"] * g["head_dim"] == g["value_dim"]
    assert g["head_dim"] == syn.D
    per_layer = bench.state_bytes_per_layer(g["v_heads"], g["channels"])
    assert per_layer == 48 * 128 * 128 * 4 + 10240 * 3 * 4
    assert round(g["layers"] * per_layer / 1e6, 1) == g["total_state_mb"]
    # the library keeps conv_state in the activation type: with bf16 activations the
    # same window holds 115.5 MB (the printed total implies 4-byte conv_state rows)
    bf16 = bench.state_bytes_per_layer(g["v_heads"], g["channels"], conv_es=2)
    assert round(g["layers"] * bf16 / 1e6, 1) == 115.5


def test_strata_geometry_limits_match_the_abi():
    g = _golden("strata_pr3226_geometry.txt")
    text = open(os.path.join(ROOT, "include", "gdn.h")).read()
    assert f"#define GDN_MAX_DRAFT {g['draft_tokens_max']}" in text
    assert f"#define GDN_HEAD_DIM {g['head_dim']}" in text
