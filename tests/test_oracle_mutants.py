"""Planted mistakes in the oracle must fail its pins.

Each case copies the oracle source, plants one plausible slip (a flipped
sign, a transposed operand, a changed reduction order, an off-by-one in the
conv_state tail ...), builds the copy on the CPU and runs the pin tests
against it: at least one pin has to fail. The real oracle is untouched.
"""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.cpp")

MUTANTS = {
    "delta_sign": ("T d = b * (v[i] - a * u);", "T d = b * (v[i] + a * u);"),
    "delta_drops_alpha": ("T d = b * (v[i] - a * u);", "T d = b * (v[i] - u);"),
    "state_transposed": ("for (int j = 0; j < D; ++j) u = u + row[j] * k[j];",
                         "for (int j = 0; j < D; ++j) u = u + S[(int64_t)j * D + i] * k[j];"),
    "output_uses_k": ("for (int j = 0; j < D; ++j) acc = acc + row[j] * q[j];",
                      "for (int j = 0; j < D; ++j) acc = acc + row[j] * k[j];"),
    "taps_reversed": ("for (int j = 0; j < KW; ++j) acc = acc + w[j] * xp_t[j];",
                      "for (int j = 0; j < KW; ++j) acc = acc + w[KW - 1 - j] * xp_t[j];"),
    "conv_drops_current_tap": ("for (int j = 0; j < KW; ++j) acc = acc + w[j] * xp_t[j];",
                               "for (int j = 0; j < KW - 1; ++j) acc = acc + w[j] * xp_t[j];"),
    "silu_without_input": ("template <class T> T silu(T y) { return y / (T(1) + std::exp(-y)); }",
                           "template <class T> T silu(T y) { return T(1) / (T(1) + std::exp(-y)); }"),
    "tail_off_by_one": ("int64_t idx = n + r;", "int64_t idx = n + r - 1;"),
    "tree_adjacent_pairs": ("T p0 = e[0] + e[4], p1 = e[1] + e[5], p2 = e[2] + e[6], p3 = e[3] + e[7];",
                            "T p0 = e[0] + e[1], p1 = e[4] + e[5], p2 = e[2] + e[3], p3 = e[6] + e[7];"),
    "eps_outside_root": ("T r = T(1) / std::sqrt(ss + eps);", "T r = T(1) / (std::sqrt(ss) + eps);"),
    "rms_not_mean": ("T ms = tree_sum_sq(o) / T(D);", "T ms = tree_sum_sq(o);"),
    "silu_sign": ("template <class T> T silu(T y) { return y / (T(1) + std::exp(-y)); }",
                  "template <class T> T silu(T y) { return y / (T(1) + std::exp(y)); }"),
    "grouping_interleaved": ("int qk_head(int h) const { return h / (Hv / Hk); }",
                             "int qk_head(int h) const { return h % Hk; }"),
    "chunk_decay_flipped": ("A[(size_t)t * chunk + s] = beta[(c0 + t) * g.Hv + h] * std::exp(G[t] - G[s])",
                            "A[(size_t)t * chunk + s] = beta[(c0 + t) * g.Hv + h] * std::exp(G[s] - G[t])"),
    "chunk_state_no_decay": ("const T gl = std::exp(G[m - 1]);", "const T gl = T(1);"),
    "gate_softplus_sign": ("alpha[i] = std::exp(-sp);", "alpha[i] = std::exp(sp);"),
    "gate_log1p_dropped": ("const T sp = x > T(0) ? x + std::log1p(std::exp(-x)) : std::log1p(std::exp(x));",
                           "const T sp = x > T(0) ? x : std::exp(x);"),
    "gate_beta_sign": ("beta[i] = T(1) / (T(1) + std::exp(-b[i]));", "beta[i] = T(1) / (T(1) + std::exp(b[i]));"),
    "commit_keeps_one_more": ("if (slot < 0 || n <= 0 || n > Tn) continue;",
                              "if (slot < 0 || n <= 0 || n > Tn) continue;\n    n = n < Tn ? n + 1 : n;"),
}

PIN_TESTS = [(name, fn) for name, fn in vars(pins).items() if name.startswith("test_")]


def _param_sets(fn):
    marks = getattr(fn, "pytestmark", [])
    for m in marks:
        if m.name == "parametrize":
            names = [n.strip() for n in m.args[0].split(",")]
            for vals in m.args[1]:
                vals = vals if len(names) > 1 else (vals,)
                yield dict(zip(names, vals))
            return
    yield {}


def _some_pin_fails():
    for name, fn in PIN_TESTS:
        for kw in _param_sets(fn):
            try:
                fn(oracle, **kw)
            except (AssertionError, ValueError, FloatingPointError):
                return name
    return None


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, mutant):
    old, new = MUTANTS[mutant]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {mutant} not found"
    mutated = src.replace(old, new, 1)
    if mutant == "commit_keeps_one_more":
        mutated = mutated.replace("const int n = n_keep[b];", "int n = n_keep[b];", 1)
    cpp = tmp_path / "mut.cpp"
    so = tmp_path / "libmut.so"
    cpp.write_text(mutated)
    subprocess.run(["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o",
                    str(so), str(cpp)], check=True)
    oracle._swap_library(str(so))
    try:
        caught = _some_pin_fails()
    finally:
        oracle._swap_library(None)
    assert caught is not None, f"no pin caught mutant {mutant}"
