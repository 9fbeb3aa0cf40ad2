"""Benchmark of the GDN token-mixing path on GB300.

Headline workload (N=1, no --workload): high-batch decode bf16 — 256 sequences,
one token each, 36 layers with q/k 16 heads and v 32 heads of 128 (C = 8192),
conv width 4, every token accepted: one step = one decode window, 36
gdn_verify_step calls with GDN_VERIFY_COMMIT_ALL (conv + SiLU + L2 norm, the
delta rule on the 18 GiB f32 state pool, z-gated RMSNorm, state and conv_state
advanced in place), through the C ABI. The same run then measures every other
workload as a further entry ("workloads"): tiny-f32, varlen-prefill-bf16
(gdn_conv_fwd + gdn_delta_prefill), spec-verify-bf16 at T = 1, 4, 8 (36 verify
launches + 1 batched commit per window) and long-prefill-bf16. Each entry has
its own roofline, kernel table, end-to-end number, clocks and CPU baseline.

metric: GDN tokens/s per layer (whole job: tokens of all ranks / max time).
--workload NAME times one workload only (also spec-verify-bf16-h48: the verify
window of one sequence with Hk = 16, Hv = 48).

Launch: python bench.py [--gpus N --steps K --warmup W] [--impl reference];
for N > 1 under torch.distributed.run, one rank per GPU, replicas of the same
workload (the path shards by sequence with no exchange: weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gated_deltanet_linear_12_gb300 import synthetic as syn  # noqa: E402

METRIC = "GDN tokens/sec per layer and achieved HBM GB/s vs GB300 peak (1 GPU)"
L2_BYTES = 129 * 1024 * 1024
D = 128


# ----------------------------------------------------------------------------- accounting
def prefill_conv_bytes(n_tok, C, n_seq_init, n_seq, es=2):
    """Algorithmic HBM bytes of gdn_conv_fwd: read x, write y, conv_w once,
    conv_state read for sequences with an initial state, written for all."""
    return 2 * n_tok * C * es + C * 4 * es + (n_seq_init + n_seq) * 3 * C * es


def prefill_delta_bytes(n_tok, C, Hv, n_seq_init, n_seq, es=2):
    """Algorithmic HBM bytes of gdn_delta_prefill: read qkv, z, alpha, beta,
    write out; state read (initial) and written (final) per sequence."""
    HvD = Hv * D
    return (n_tok * (C * es + 2 * HvD * es + 2 * Hv * 4)
            + (n_seq_init + n_seq) * Hv * D * D * 4)


def prefill_delta_flops(n_tok, Hv):
    """Algorithmic FLOPs of the chunked form per token-head: five 64x64x128
    intra-chunk products (k.k, q.k, Tinv-applied values and keys, scores x
    deltas) = 81,920 FLOP and three 64x128x128 state products = 98,304 FLOP."""
    return n_tok * Hv * (5 * 64 * 128 * 2 + 3 * 128 * 128 * 2)


def window_bytes(B, T, Hv, C, L, n_keep, decode=False, lazy=False):
    """Algorithmic HBM bytes of one window over L layers (bf16 activations, f32
    state and gates): "verify" for the verify launches (decode: the commit-all
    verify, which also writes S and conv_state; lazy: the verify that first
    commits the previous window's n_keep[b] tokens) and "commit" for the batched
    commit of the accepted prefixes n_keep[b]."""
    per_seq_state = Hv * D * D * 4
    conv_rows = 3 * C * 2
    drafts = B * T * (C * 2 + 2 * Hv * D * 2 + 2 * Hv * 4) + C * 4 * 2   # x, z, out, gates, conv_w
    accepted = [int(n) for n in n_keep if n > 0]
    if lazy:
        verify = B * per_seq_state + B * conv_rows + drafts + sum(
            per_seq_state + conv_rows + n * (C * 2 + 2 * Hv * 4) for n in accepted)
        return {"verify": L * verify, "commit": 0}
    rw = 2 if decode else 1
    verify = B * per_seq_state * rw + B * conv_rows * rw + drafts
    commit = 0 if decode else sum(2 * per_seq_state + 2 * conv_rows + n * (C * 2 + 2 * Hv * 4)
                                  + C * 4 * 2 for n in accepted)
    return {"verify": L * verify, "commit": L * commit}


def state_bytes_per_layer(Hv, C, dv=D, dk=D, conv_rows=3, state_es=4, conv_es=4):
    """Bytes of one layer's recurrent state plus conv_state for one sequence."""
    return Hv * dv * dk * state_es + C * conv_rows * conv_es


def prefill_roofline(kernel, flops, nbytes, ms, peaks, peak_src, traffic):
    """Roofline entry of a prefill launch of `flops` algorithmic FLOPs and
    `nbytes` algorithmic HBM bytes that took `ms`. The binding roofline is the one
    with the longer floor: the bytes at the HBM peak, or the FLOPs at the peak of
    the unit the products run on (tensor cores for bf16, the FP32 pipe for f32).
    Both fractions are reported."""
    s = ms * 1e-3
    gbs, tflops = nbytes / s / 1e9, flops / s / 1e12
    if kernel == "prefill_tc_kernel":
        c_bound, c_peak = "tensor", peaks.get("bf16_tflops", 1920.0)
        c_src = f"{peak_src} (MEASURED_PEAKS.json bf16_tflops, burst)"
    else:
        mhz = peaks.get("sm_max_mhz", 2070.0)
        c_bound, c_peak = "alu", round(fp32_alu_peak_tflops(mhz), 1)
        c_src = f"derived: 152 SMs x 128 FP32 lanes x 2 FLOP x {mhz:.0f} MHz"
    floor_hbm_us = nbytes / (peaks["hbm_gbs"] * 1e9) * 1e6
    floor_c_us = flops / (c_peak * 1e12) * 1e6
    common = {"algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": nbytes,
              "traffic_per": "launch (ncu, one pass)",
              "floor_us": {"hbm": round(floor_hbm_us, 2), c_bound: round(floor_c_us, 2)},
              "hbm_gbs": round(gbs, 1), "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
              f"{c_bound}_tflops": round(tflops, 3), f"{c_bound}_frac": round(tflops / c_peak, 4)}
    if floor_hbm_us >= floor_c_us:
        return {"kernel": kernel, "bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": traffic,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)", **common}
    return {"kernel": kernel, "bound": c_bound, "achieved": round(tflops, 3), "peak": c_peak,
            "unit": "TFLOP/s", "frac": round(tflops / c_peak, 4),
            "traffic": traffic if c_bound == "tensor" else None, "peak_source": c_src, **common}


def gates_note(gates):
    return ("raw projections; the gate step runs inside the kernels" if gates == "raw"
            else "activated alpha, beta inputs")


def max_over_ranks(value, device, world):
    """The largest value over the ranks (every rank gets it): with independent
    replicas the job is done when the slowest one is."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, ms_max):
    """Units processed by all ranks per second, from the slowest rank's time."""
    return units_per_rank * world / (ms_max * 1e-3)


def fp32_alu_peak_tflops(sm_mhz, n_sm=152, lanes=128):
    """FP32 FMA peak: SMs x FP32 lanes per SM x 2 FLOP x clock."""
    return n_sm * lanes * 2 * sm_mhz * 1e6 / 1e12


# ----------------------------------------------------------------------------- helpers
KERNEL_SOURCES = {
    "prefill_tc_kernel": ["gated_deltanet_linear_12_gb300/csrc/prefill_tc.cu",
                          "gated_deltanet_linear_12_gb300/csrc/tc.cuh",
                          "gated_deltanet_linear_12_gb300/csrc/common.cuh"],
    "conv_fwd_kernel": ["gated_deltanet_linear_12_gb300/csrc/conv.cu",
                        "gated_deltanet_linear_12_gb300/csrc/common.cuh"],
    "step_kernel": ["gated_deltanet_linear_12_gb300/csrc/step.cu",
                    "gated_deltanet_linear_12_gb300/csrc/common.cuh"],
    "lazy_kernel": ["gated_deltanet_linear_12_gb300/csrc/step.cu",
                    "gated_deltanet_linear_12_gb300/csrc/common.cuh"],
    "verify_kernel": ["gated_deltanet_linear_12_gb300/csrc/verify.cu",
                      "gated_deltanet_linear_12_gb300/csrc/tc.cuh",
                      "gated_deltanet_linear_12_gb300/csrc/common.cuh"],
}


def source_hash(kernel):
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu record of this kernel and
    workload, or None when the kernel's source changed since the capture."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 3 and not line.startswith("#") and parts[0] == f"{kernel}/{workload}":
                return int(parts[2]) if parts[1] == source_hash(kernel) else None
    return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "sm_max_mhz": 2070.0}, "fallback"


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        # the raw samples (a CSV); GDN_CLOCK_LOG_DIR keeps them somewhere of the user's choice
        log_dir = os.environ.get("GDN_CLOCK_LOG_DIR") or tempfile.gettempdir()
        self.path = os.path.join(log_dir, f"gdn_bench_clocks_gpu{gpu_index}_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- workloads
class PrefillWorkload:
    """One layer's varlen prefill; inputs resident on the device."""

    def __init__(self, name, torch, G, device, gates="activated"):
        self.name, self.torch, self.G, self.dev = name, torch, G, device
        self.gates = gates
        inp = syn.workload_prefill(name, gate_form="raw" if gates == "raw" else None)
        self.inp = inp
        self.act = torch.bfloat16 if inp["act"] == "bf16" else torch.float32
        t = lambda a: self._dev(a)
        self.x = t(inp["x"])
        self.y = torch.empty_like(self.x)
        self.conv_w = t(inp["conv_w"])
        self.cs0 = t(inp["conv_state"])
        self.cs = self.cs0.clone()
        self.S0 = t(inp["state"])
        self.S = self.S0.clone()
        self.alpha, self.beta, self.z = t(inp["alpha"]), t(inp["beta"]), t(inp["z"])
        self.norm_w = t(inp["norm_w"])
        self.slot, self.cu = t(inp["slot_idx"]), t(inp["cu_seqlens"])
        self.hic, self.his = t(inp["has_init_conv"]), t(inp["has_init_state"])
        self.out = torch.empty(inp["n_tok"], inp["Hv"] * D, dtype=self.act, device=device)
        self.cfg = G.make_config(inp["Hk"], inp["Hv"], self.act, self.S.shape[0],
                                 gates=G.GDN_GATES_RAW if gates == "raw" else G.GDN_GATES_ACTIVATED)
        self.tokens = int(inp["n_tok"])
        es = 2 if inp["act"] == "bf16" else 4
        n_init_c = int(inp["has_init_conv"].sum())
        n_init_s = int(inp["has_init_state"].sum())
        self.bytes = {"conv": prefill_conv_bytes(self.tokens, inp["C"], n_init_c, inp["n_seq"], es),
                      "prefill": prefill_delta_bytes(self.tokens, inp["C"], inp["Hv"], n_init_s,
                                                     inp["n_seq"], es)}
        self.flops = {"prefill": prefill_delta_flops(self.tokens, inp["Hv"])}
        self.launches_per_step = 2

    def _dev(self, a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return self.torch.from_numpy(a.view(np.int16)).to(self.dev).view(self.torch.bfloat16)
        return self.torch.from_numpy(a).to(self.dev)

    def reset(self):
        self.cs.copy_(self.cs0)
        self.S.copy_(self.S0)

    def step(self, ev=None):
        G = self.G
        if ev:
            ev[0].record()
        G.gdn_conv_fwd(self.cfg, self.x, self.y, self.conv_w, self.cs, self.slot, self.cu, self.hic)
        if ev:
            ev[1].record()
        G.gdn_delta_prefill(self.cfg, self.y, self.alpha, self.beta, self.z, self.norm_w, self.out,
                            self.S, self.slot, self.cu, self.his)
        if ev:
            ev[2].record()

    # end-to-end: host inputs -> device, step, result -> host (pinned buffers)
    def setup_e2e(self):
        torch = self.torch
        self.h_in = [a.cpu().pin_memory() for a in (self.x, self.alpha, self.beta, self.z)]
        self.d_in = [self.x, self.alpha, self.beta, self.z]
        self.h_out = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self.h2d = sum(a.numel() * a.element_size() for a in self.h_in)
        self.d2h = self.h_out.numel() * self.h_out.element_size()

    def step_e2e(self):
        for h, d in zip(self.h_in, self.d_in):
            d.copy_(h, non_blocking=True)
        self.step()
        self.h_out.copy_(self.out, non_blocking=True)

    def config(self):
        inp = self.inp
        return {"workload": self.name, "n_seq": int(inp["n_seq"]), "tokens": self.tokens,
                "lens": [int(v) for v in inp["lens"]], "qk_heads": int(inp["Hk"]),
                "v_heads": int(inp["Hv"]), "head_dim": D, "conv_width": 4, "channels": int(inp["C"]),
                "chunk": 64, "state_dtype": "f32", "act_dtype": inp["act"],
                "gates": gates_note(self.gates),
                "l2": "flush 256 MiB between timed steps"}


class StepWorkload:
    """Verify windows (spec-verify-bf16: per window 36 verify calls of one launch each, then one
    batched commit of the accepted prefixes of all 36 layers) or decode
    (decode-bf16: 36 verify launches with every token accepted). Each layer has
    its own conv_state and state pools; inputs are seeded and generated on the
    device (standard normals; alpha = exp(-softplus(N)), beta = sigmoid(N))."""

    LAYERS = 36

    def __init__(self, name, torch, G, device, T=None, gates="activated", lazy=False, batch=None):
        self.name, self.torch, self.G, self.dev = name, torch, G, device
        self.gates = gates
        raw = gates == "raw"
        # lazy: each verify launch first commits the previous window's accepted prefix
        self.lazy = lazy and name != "decode-bf16"
        decode = name == "decode-bf16"
        self.decode = decode
        h48 = name == "spec-verify-bf16-h48"
        self.B = batch or (256 if decode else 1 if h48 else 32)
        self.T = 1 if decode else (T or 8)
        self.Hk, self.Hv = 16, 48 if h48 else 32
        self.C = (2 * self.Hk + self.Hv) * D
        B, T, Hv, C, L = self.B, self.T, self.Hv, self.C, self.LAYERS
        g = torch.Generator(device=device)
        g.manual_seed(syn.seed_of(name) + T)
        bf = torch.bfloat16
        self.n_slots = B
        rn = lambda *shape, dt=torch.float32: torch.randn(*shape, generator=g, device=device,
                                                          dtype=torch.float32).to(dt)
        self.layers = []
        for _ in range(L):
            lay = dict(x=rn(B, T, C, dt=bf), conv_w=(rn(C, 4) * 0.5).to(bf),
                       conv_state=rn(B, 3, C, dt=bf), state=rn(B, Hv, D, D),
                       alpha=rn(B, T, Hv) if raw else torch.exp(-torch.nn.functional.softplus(rn(B, T, Hv))),
                       beta=rn(B, T, Hv) if raw else torch.sigmoid(rn(B, T, Hv)),
                       z=rn(B, T, Hv * D, dt=bf))
            if self.lazy:                                   # the previous window's drafts
                lay.update(px=rn(B, T, C, dt=bf),
                           palpha=rn(B, T, Hv) if raw else torch.exp(-torch.nn.functional.softplus(rn(B, T, Hv))),
                           pbeta=rn(B, T, Hv) if raw else torch.sigmoid(rn(B, T, Hv)))
            self.layers.append(lay)
        self.norm_w = (1 + 0.1 * rn(D)).contiguous()
        self.slot = torch.randperm(B, generator=g, device=device).to(torch.int32)
        self.n_keep = torch.randint(0, T + 1, (B,), generator=g, device=device, dtype=torch.int32)
        self.out = torch.empty(B, T, Hv * D, dtype=bf, device=device)
        self.cfg = G.make_config(self.Hk, self.Hv, bf, self.n_slots,
                                 gates=G.GDN_GATES_RAW if raw else G.GDN_GATES_ACTIVATED)
        self.views = G.make_layer_views([{k: l[k] for k in ("x", "alpha", "beta", "conv_w",
                                                             "conv_state", "state")}
                                         for l in self.layers], device)
        self.tokens = B * T                                 # per layer per step
        # read-only verify: one cooperative launch per layer, then one commit launch
        self.launches_per_step = L if (decode or self.lazy) else L + 1
        self.ws = None if decode else G.verify_workspace(self.cfg, B, T, device)
        self.bytes = window_bytes(B, T, Hv, C, L, self.n_keep.cpu().numpy(), decode=decode,
                                  lazy=self.lazy)

    def reset(self):
        pass                                                # state evolution does not change work

    def verify_layers(self):
        G = self.G
        if self.lazy:
            for lay in self.layers:
                G.gdn_verify_step_lazy(self.cfg, lay["px"], lay["palpha"], lay["pbeta"], self.n_keep,
                                       lay["x"], lay["conv_w"], lay["conv_state"], lay["state"],
                                       lay["alpha"], lay["beta"], lay["z"], self.norm_w, self.out,
                                       self.slot)
            return
        for lay in self.layers:
            G.gdn_verify_step(self.cfg, lay["x"], lay["conv_w"], lay["conv_state"], lay["state"],
                              lay["alpha"], lay["beta"], lay["z"], self.norm_w, self.out, self.slot,
                              commit_all=self.decode, workspace=self.ws)

    def commit(self):
        if not self.decode and not self.lazy:
            self.G.gdn_commit_layers(self.cfg, self.views, self.LAYERS, self.slot, self.n_keep, self.T)

    def capture(self):
        """The window's launches as two CUDA graphs (the 36 verify calls, the
        commit), as a serving loop replays them: the per-call host cost of the
        C ABI (about 15 us through the Python binding) then stays off the GPU's
        timeline. Captured through the same public calls."""
        torch = self.torch
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        self.g_verify, self.g_commit = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(self.g_verify, stream=s):
                self.verify_layers()
            if not self.lazy:                           # lazy: the commit rides on the verify
                with torch.cuda.graph(self.g_commit, stream=s):
                    self.commit()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()

    def step(self, ev=None):
        graphs = hasattr(self, "g_verify")
        if ev:
            ev[0].record()
        self.g_verify.replay() if graphs else self.verify_layers()
        if ev:
            ev[1].record()
        if not self.lazy:
            self.g_commit.replay() if graphs else self.commit()
        if ev:
            ev[2].record()

    def setup_e2e(self):
        torch = self.torch
        self.h_x = [l["x"].cpu().pin_memory() for l in self.layers]
        self.h_out = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self.h2d = sum(a.numel() * a.element_size() for a in self.h_x)
        self.d2h = self.h_out.numel() * self.h_out.element_size()

    def step_e2e(self):
        """Direct calls through the public API (no graph), host copies included."""
        for h, l in zip(self.h_x, self.layers):
            l["x"].copy_(h, non_blocking=True)
        self.verify_layers()
        self.commit()
        self.h_out.copy_(self.out, non_blocking=True)

    def config(self):
        return {"workload": self.name, "batch": self.B, "draft_tokens": self.T,
                "layers": self.LAYERS, "qk_heads": self.Hk, "v_heads": self.Hv, "head_dim": D,
                "channels": self.C, "state_dtype": "f32", "act_dtype": "bf16",
                "n_keep": "uniform in [0, T]" if not self.decode else "all",
                "window": ("lazy: each verify launch commits the previous window's accepted prefix"
                           if self.lazy else "verify launches, then one batched commit"),
                "gates": gates_note(self.gates),
                "launch": "CUDA graphs of the window's public calls (value); direct calls (e2e)",
                "l2": "state pools of all layers exceed L2; flush 256 MiB between timed steps"}


# ----------------------------------------------------------------------------- CPU baseline
def host_info():
    """The host the CPU baseline ran on: logical CPUs and the CPU model."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        import platform
        model = platform.processor() or platform.machine()
    return {"nproc": os.cpu_count(), "cpu_model": model}


def cpu_baseline(name, max_tokens=None, gates="activated"):
    """The oracle as it stands (single thread) on the prefill workload: its
    sequences in full, or the first max_tokens tokens of them; conv (+ the gate
    step for raw gates) + token-by-token recurrence in f64."""
    import oracle as orc
    raw = gates == "raw"
    inp = syn.workload_prefill(name, gate_form="raw" if raw else None)
    lens, cu = inp["lens"], inp["cu_seqlens"]
    cap = int(inp["n_tok"]) if max_tokens is None else max_tokens
    keep, tot = [], 0
    for s in range(inp["n_seq"]):
        n = int(min(lens[s], cap - tot))
        if n <= 0:
            break
        keep.append((s, n))
        tot += n
    rows = np.concatenate([np.arange(cu[s], cu[s] + n) for s, n in keep])
    cu2 = np.concatenate([[0], np.cumsum([n for _, n in keep])]).astype(np.int32)
    ss = [s for s, _ in keep]
    t0 = time.perf_counter()
    y, _ = orc.conv_fwd(inp["x"][rows], inp["conv_w"], inp["conv_state"], inp["slot_idx"][ss], cu2,
                        inp["has_init_conv"][ss], inp["Hk"], inp["Hv"])
    if inp["act"] == "bf16":
        y = orc.round_bf16(y)
    al, be = inp["alpha"][rows], inp["beta"][rows]
    if raw:
        al, be = orc.gates(al, be)
    orc.prefill(y, al, be, inp["z"][rows], inp["norm_w"],
                inp["state"], inp["slot_idx"][ss], cu2, inp["has_init_state"][ss], inp["Hk"],
                inp["Hv"])
    dt = time.perf_counter() - t0
    full = tot == int(inp["n_tok"])
    what = (f"the whole {name} workload ({tot} tokens, {len(keep)} sequences)" if full else
            f"first {tot} tokens of {len(keep)} sequence(s) of the {name} workload")
    return {"value": tot / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{what}, conv + {'gate step + ' if raw else ''}token-by-token recurrence "
                      f"in f64, {dt:.1f} s", "host": host_info()}


def cpu_baseline_window(name, T, n_seq=None, gates="activated"):
    """The oracle on one layer of a verify / decode window: n_seq sequences
    (default: the workload's whole batch) verified, then the accepted prefix
    committed (decode: the commit-all verify), as tokens per second per layer."""
    import oracle as orc
    decode = name == "decode-bf16"
    h48 = name == "spec-verify-bf16-h48"
    Hv = 48 if h48 else 32
    T = 1 if decode else T
    if n_seq is None:
        n_seq = 256 if decode else 1 if h48 else 32
    raw = gates == "raw"
    inp = syn.verify_inputs(n_seq, T, 16, Hv, "bf16", seed=syn.seed_of(name) + T,
                            gate_form="raw" if raw else "softplus")
    t0 = time.perf_counter()
    al, be = (orc.gates(inp["alpha"], inp["beta"]) if raw else (inp["alpha"], inp["beta"]))
    orc.verify(inp["x"], inp["conv_w"], inp["conv_state"], inp["state"], al, be, inp["z"],
               inp["norm_w"], inp["slot_idx"], 16, Hv, commit_all=decode)
    if not decode:
        orc.commit(inp["x"], al, be, inp["conv_w"], inp["conv_state"], inp["state"],
                   inp["slot_idx"], inp["n_keep"], 16, Hv)
    dt = time.perf_counter() - t0
    return {"value": n_seq * T / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"one layer of the {name} window in full ({n_seq} sequences x {T} tokens), "
                      f"{'gate step + ' if raw else ''}verify{'' if decode else ' + commit'} in f64, "
                      f"{dt:.2f} s", "host": host_info()}


# ----------------------------------------------------------------------------- main
WINDOWS = ("spec-verify-bf16", "spec-verify-bf16-h48", "decode-bf16")
# The default run: the largest single-GPU workload as the headline, then every
# other workload of the benchmark as a further entry of the same line.
HEADLINE = "decode-bf16"
EXTRAS = [("tiny-f32", None), ("varlen-prefill-bf16", None), ("spec-verify-bf16", 1),
          ("spec-verify-bf16", 4), ("spec-verify-bf16", 8), ("long-prefill-bf16", None)]
# CPU-baseline sample per prefill workload (None: the whole workload)
CPU_PREFILL_TOKENS = {"tiny-f32": None, "varlen-prefill-bf16": None, "long-prefill-bf16": 4096}


def run_workload(name, T, args, torch, G, dev, world, barrier, flush, lazy=False, steps=None,
                 cpu=True, batch=None):
    """Times one workload (value: device time of the step, CUDA events on the
    launching stream; e2e: the same calls with host copies). Returns the fields
    of its JSON entry; every rank returns, rank 0's is printed."""
    steps = steps or args.steps
    if name in WINDOWS:
        W = StepWorkload(name, torch, G, dev, T=T, gates=args.gates, lazy=lazy, batch=batch)
    else:
        W = PrefillWorkload(name, torch, G, dev, gates=args.gates)
    for _ in range(max(args.warmup, 3)):
        W.reset()
        W.step()
    torch.cuda.synchronize()
    if isinstance(W, StepWorkload):
        W.capture()
        for _ in range(2):
            W.step()
        torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    time.sleep(0.3)
    barrier()
    t_wall = time.perf_counter()
    for k in range(steps):
        W.reset()
        flush.fill_(float(k))
        W.step(evs[k])
    barrier()
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    conv_ms = [evs[k][0].elapsed_time(evs[k][1]) for k in range(steps)]
    pf_ms = [evs[k][1].elapsed_time(evs[k][2]) for k in range(steps)]
    step_ms = [c + p for c, p in zip(conv_ms, pf_ms)]
    ms = statistics.mean(step_ms)
    ms_max = max_over_ranks(ms, dev, world)

    # end-to-end through the public API with host buffers
    W.setup_e2e()
    for _ in range(3):
        W.reset()
        W.step_e2e()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_ms = []
    for k in range(steps):
        W.reset()
        flush.fill_(float(k))
        e0.record()
        W.step_e2e()
        e1.record()
        e1.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    e2e_max = max_over_ranks(statistics.mean(e2e_ms), dev, world)

    peaks, peak_src = load_peaks()
    a_avg, b_avg = statistics.mean(conv_ms), statistics.mean(pf_ms)
    if isinstance(W, StepWorkload):
        vk = "step_kernel" if W.decode else "lazy_kernel" if W.lazy else "verify_kernel"
        names = (f"{vk} ({'decode' if W.decode else 'commit + verify' if W.lazy else 'verify'})",
                 "step_kernel (commit)")
        ka = {"ms": round(a_avg, 4), "bytes": W.bytes["verify"],
              "GB/s": round(W.bytes["verify"] / (a_avg * 1e-3) / 1e9, 1)}
        ka["frac_hbm"] = round(ka["GB/s"] / peaks["hbm_gbs"], 4)
        kernels = {names[0]: ka}
        if not W.decode and not W.lazy:
            kb = {"ms": round(b_avg, 4), "bytes": W.bytes["commit"],
                  "GB/s": round(W.bytes["commit"] / max(b_avg, 1e-9) / 1e6, 1)}
            kb["frac_hbm"] = round(kb["GB/s"] / peaks["hbm_gbs"], 4)
            kernels[names[1]] = kb
        roof = {"kernel": names[0] + f", {W.LAYERS} launches", "bound": "hbm",
                "achieved": ka["GB/s"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ka["frac_hbm"], "traffic": ncu_traffic(vk, W.name + f"/T{W.T}"),
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                "algorithmic_bytes_per_window": W.bytes["verify"],
                "algorithmic_bytes_per_launch": W.bytes["verify"] // W.LAYERS,
                "traffic_per": "launch (ncu, one pass)"}
        value = whole_job_rate(W.tokens * W.LAYERS, world, ms_max)
    else:
        pf_tflops = W.flops["prefill"] / (b_avg * 1e-3) / 1e12
        pf_gbs = W.bytes["prefill"] / (b_avg * 1e-3) / 1e9
        conv_gbs = W.bytes["conv"] / (a_avg * 1e-3) / 1e9
        pf_name = "prefill_tc_kernel" if W.inp["act"] == "bf16" else "prefill_ffma_kernel"
        if b_avg >= a_avg:
            roof = prefill_roofline(pf_name, W.flops["prefill"], W.bytes["prefill"], b_avg, peaks,
                                    peak_src, ncu_traffic(pf_name, W.name))
        else:
            roof = {"kernel": "conv_fwd_kernel", "bound": "hbm", "achieved": round(conv_gbs, 1),
                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": round(conv_gbs / peaks["hbm_gbs"], 4),
                    "traffic": ncu_traffic("conv_fwd_kernel", W.name),
                    "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                    "algorithmic_bytes_per_launch": W.bytes["conv"], "traffic_per": "launch (ncu, one pass)"}
        kernels = {
            "conv_fwd_kernel": {"ms": round(a_avg, 4), "bytes": W.bytes["conv"],
                                "GB/s": round(conv_gbs, 1),
                                "frac_hbm": round(conv_gbs / peaks["hbm_gbs"], 4)},
            pf_name: {"ms": round(b_avg, 4), "bytes": W.bytes["prefill"],
                      "GB/s": round(pf_gbs, 1), "frac_hbm": round(pf_gbs / peaks["hbm_gbs"], 4),
                      "TFLOP/s": round(pf_tflops, 3)},
        }
        value = whole_job_rate(W.tokens, world, ms_max)
    e2e_val = value * ms_max / e2e_max
    entry = {
        "value": round(value, 1), "unit": "tokens/s", "steps": steps,
        "ms_per_step": round(ms_max, 4), "ms_min": round(min(step_ms), 4),
        "ms_max": round(max(step_ms), 4), "dtype": "f32" if name == "tiny-f32" else "bf16",
        "config": W.config(), "roofline": roof, "kernels": kernels,
        "e2e": {"value": round(e2e_val, 1), "unit": "tokens/s", "h2d_bytes_per_step": W.h2d,
                "d2h_bytes_per_step": W.d2h},
        "gpu_launches": W.launches_per_step * steps,
        "clocks": {k: clk.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "wall_s_timed_region": round(t_wall, 3),
    }
    del W
    torch.cuda.empty_cache()
    if world == 1 and cpu and not args.no_cpu_baseline and int(os.environ.get("RANK", "0")) == 0:
        if name in WINDOWS:
            entry["cpu_baseline"] = cpu_baseline_window(name, T or 8, gates=args.gates)
        else:
            entry["cpu_baseline"] = cpu_baseline(name, max_tokens=CPU_PREFILL_TOKENS.get(name, 4096),
                                                 gates=args.gates)
    return entry


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=None,
                    help=f"one workload only (default: {HEADLINE} as the headline, then the others)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--T", type=int, default=8, help="draft tokens of spec-verify-bf16")
    ap.add_argument("--batch", type=int, default=None,
                    help="sequences of the --workload window (decode-bf16, spec-verify-bf16): "
                         "a smaller case of the same kernels for profiling; not a bench line")
    ap.add_argument("--lazy", action="store_true",
                    help="verify windows: fold each window's commit into the next window's verify")
    ap.add_argument("--gates", default="activated", choices=["activated", "raw"],
                    help="raw: alpha / beta inputs are raw projections and the kernels apply "
                         "the gate step as they read them")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return reference_arm(args, rank, world)

    import torch
    import torch.distributed as dist
    from gated_deltanet_linear_12_gb300 import build as _build, gdn as G
    if not os.path.exists(_build.LIB):
        _build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    name = args.workload or HEADLINE
    head = run_workload(name, args.T, args, torch, G, dev, world, barrier, flush, lazy=args.lazy,
                        batch=args.batch)
    extras = {}
    if args.workload is None:
        for wname, T in EXTRAS:
            key = wname if T is None else f"{wname}/T{T}"
            extras[key] = run_workload(wname, T, args, torch, G, dev, world, barrier, flush,
                                       steps=min(args.steps, 20))
    if rank == 0:
        line = {"metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": max(args.warmup, 3),
                "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic"}
        line.update({k: v for k, v in head.items() if k not in line and k != "steps"})
        if extras:
            line["workloads"] = extras
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def reference_arm(args, rank, world):
    """The oracle as the reference arm: each step is one bounded sample of the
    workload run by the single-threaded CPU oracle."""
    if rank != 0:
        return 0
    import oracle as orc
    orc.build()
    for _ in range(args.warmup):
        pass                                      # the oracle has no warm-up state
    name = args.workload or HEADLINE
    window = name in WINDOWS
    n_seq = 16                                   # sequences of one layer per step
    times, toks = [], 0
    line0 = None
    for _ in range(args.steps):
        cb = (cpu_baseline_window(name, args.T, n_seq=n_seq, gates=args.gates) if window
              else cpu_baseline(name, max_tokens=512, gates=args.gates))
        times.append(1.0 / cb["value"])
        line0 = cb
    tps = 1.0 / statistics.mean(times)
    per_step = (n_seq * (1 if name == "decode-bf16" else args.T)) if window else 512
    line = {"impl": "reference", "metric": METRIC, "value": round(tps, 2), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per_step / tps * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": name, "gates": gates_note(args.gates),
                       "sample": line0["sample"] if line0 else ""},
            "cpu_baseline": {"value": round(tps, 2), "unit": "tokens/s", "cores": 1,
                             "kind": "oracle", "sample": line0["sample"] if line0 else "",
                             "host": host_info()},
            "e2e": {"value": round(tps, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
