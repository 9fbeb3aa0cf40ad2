"""Seeded synthetic inputs for the Gated DeltaNet token-mixing path.

This module is shared by the tests, the benchmark and the CPU oracle's
callers. It draws random numbers and packs them into the layouts the path
uses; it performs none of the path's arithmetic (no convolution, activation,
normalisation or recurrence). Gate values alpha and beta are drawn in their
activated form (the workloads' distribution, alpha = exp(-softplus(N)) and
beta = sigmoid(N), written here with numpy as an input recipe), or, with
gate_form "raw", as the raw projections a, b ~ N(0, 1) that the library's gate
step (and the oracle's, independently) turns into that same distribution.

Layouts (row-major, head_dim d = 128, conv width 4):
  qkv / x       [n_tok][C], C = (2*Hk + Hv) * d, channels packed [q | k | v]
  conv_w        [C][4], tap 3 multiplies the current token
  conv_state    [n_slots][3][C], oldest row first
  state (S)     [n_slots][Hv][d (value rows)][d (key columns)] float32
  alpha, beta   [n_tok][Hv] float32
  z, out        [n_tok][Hv*d]
Activations in "bf16" are returned as uint16 bit patterns (round to nearest
even from float32); "f32" activations are float32 arrays.

Workloads (names used across the repository):
  tiny-f32              1 sequence of 64 tokens, Hk=2, Hv=4 (C=1024), f32
  varlen-prefill-bf16   8 sequences, lengths uniform in [1, 2048], Hk=16, Hv=32
  spec-verify-bf16      batch 32, T = 1..8 draft tokens, 36 layers
  long-prefill-bf16     4 sequences x 16384 tokens
  decode-bf16           batch 256, T = 1, 36 layers
  spec-verify-bf16-h48  one sequence, T = 1..8, Hk=16, Hv=48 (C=10240), 36 layers
"""
from __future__ import annotations

import numpy as np

D = 128
KW = 4

SEED_BASE = 0x6D6E0000

WORKLOADS = [
    "tiny-f32",
    "varlen-prefill-bf16",
    "spec-verify-bf16",
    "long-prefill-bf16",
    "decode-bf16",
    "spec-verify-bf16-h48",
]


def seed_of(name: str) -> int:
    return SEED_BASE + WORKLOADS.index(name)


# ---------------------------------------------------------------- bf16 bits
def f32_to_bf16_bits(a) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32)
            << np.uint32(16)).view(np.float32)


def to_act(a, act: str) -> np.ndarray:
    """Store float32 values in the activation type ('f32' or 'bf16' bits)."""
    if act == "f32":
        return np.ascontiguousarray(a, dtype=np.float32)
    if act == "bf16":
        return f32_to_bf16_bits(a)
    raise ValueError(act)


def act_to_f32(a, act: str) -> np.ndarray:
    return np.asarray(a, np.float32) if act == "f32" else bf16_bits_to_f32(a)


def channels(Hk: int, Hv: int) -> int:
    return (2 * Hk + Hv) * D


# ---------------------------------------------------------------- gates
def _gates(rng, shape, form: str):
    if form == "uniform":          # alpha ~ U(0.9, 1), beta ~ U(0, 1)
        a = rng.uniform(0.9, 1.0, size=shape).astype(np.float32)
        b = rng.uniform(0.0, 1.0, size=shape).astype(np.float32)
    elif form == "raw":            # raw projections a, b ~ N(0, 1) for the gate step
        a = rng.standard_normal(shape).astype(np.float32)
        b = rng.standard_normal(shape).astype(np.float32)
    elif form == "softplus":       # alpha = exp(-softplus(N)), beta = sigmoid(N)
        na = rng.standard_normal(shape)
        nb = rng.standard_normal(shape)
        a = np.exp(-np.logaddexp(0.0, na)).astype(np.float32)
        b = (1.0 / (1.0 + np.exp(-nb))).astype(np.float32)
    else:
        raise ValueError(form)
    return a, b


def _normal(rng, shape, sigma=1.0):
    return (rng.standard_normal(shape, dtype=np.float32) * np.float32(sigma))


# ---------------------------------------------------------------- prefill
def prefill_inputs(lens, Hk, Hv, act, *, seed, init_mask=None, gate_form="softplus",
                   init_conv=None, init_state=None, n_slots=None, slot_perm=True):
    """Inputs of one layer's varlen prefill (conv, then the chunked recurrence).

    lens        sequence lengths (tokens)
    init_mask   per sequence: 1 = has an initial conv_state and state S
    init_conv / init_state  override init_mask for the conv or the state alone
    Returns a dict of numpy arrays; slot_idx maps sequences onto pool slots.
    """
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int64)
    n_seq = len(lens)
    C = channels(Hk, Hv)
    n_tok = int(lens.sum())
    cu = np.zeros(n_seq + 1, np.int32)
    cu[1:] = np.cumsum(lens)
    if init_mask is None:
        init_mask = np.zeros(n_seq, np.uint8)
    init_mask = np.asarray(init_mask, np.uint8)
    has_conv = init_mask if init_conv is None else np.asarray(init_conv, np.uint8)
    has_state = init_mask if init_state is None else np.asarray(init_state, np.uint8)
    n_slots = n_seq + 2 if n_slots is None else n_slots
    slots = rng.permutation(n_slots)[:n_seq].astype(np.int32) if slot_perm \
        else np.arange(n_seq, dtype=np.int32)

    x = _normal(rng, (n_tok, C))
    conv_w = _normal(rng, (C, KW), 0.5)          # N(0, 0.25): variance 0.25
    conv_state = _normal(rng, (n_slots, KW - 1, C))
    state = _normal(rng, (n_slots, Hv, D, D))
    alpha, beta = _gates(rng, (n_tok, Hv), gate_form)
    z = _normal(rng, (n_tok, Hv * D))
    norm_w = (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    return dict(
        lens=lens, cu_seqlens=cu, n_seq=n_seq, n_tok=n_tok, C=C, Hk=Hk, Hv=Hv, act=act,
        slot_idx=slots, has_init_conv=has_conv, has_init_state=has_state,
        x=to_act(x, act), conv_w=to_act(conv_w, act),
        conv_state=to_act(conv_state, act), state=state,
        alpha=alpha, beta=beta, z=to_act(z, act), norm_w=norm_w,
    )


def workload_prefill(name: str, *, seed=None, gate_form=None):
    """gate_form None: the workload's own; "raw": raw projections for the gate step."""
    seed = seed_of(name) if seed is None else seed
    gf = gate_form or "softplus"
    if name == "tiny-f32":
        # one sequence of 64 tokens; random conv_state read, zero initial S
        return prefill_inputs([64], 2, 4, "f32", seed=seed, init_conv=[1], init_state=[0],
                              gate_form=gate_form or "uniform")
    if name == "varlen-prefill-bf16":
        rng = np.random.default_rng(seed ^ 0x5EED)
        lens = rng.integers(1, 2049, size=8)
        mask = np.array([i % 2 for i in range(8)], np.uint8)   # odd sequences carry state
        return prefill_inputs(lens, 16, 32, "bf16", seed=seed, init_mask=mask, gate_form=gf)
    if name == "long-prefill-bf16":
        return prefill_inputs([16384] * 4, 16, 32, "bf16", seed=seed,
                              init_mask=np.zeros(4, np.uint8), gate_form=gf)
    raise ValueError(name)


# ---------------------------------------------------------------- verify / decode
def verify_inputs(B, T, Hk, Hv, act, *, seed, n_slots=None, gate_form="softplus",
                  pad_slots=0):
    """One layer of a speculative-verify window: T draft tokens per sequence.

    pad_slots   number of trailing batch entries given slot -1 (padding)
    """
    rng = np.random.default_rng(seed)
    C = channels(Hk, Hv)
    n_slots = B + 3 if n_slots is None else n_slots
    slots = rng.permutation(n_slots)[:B].astype(np.int32)
    if pad_slots:
        slots[B - pad_slots:] = -1
    x = _normal(rng, (B, T, C))
    conv_w = _normal(rng, (C, KW), 0.5)
    conv_state = _normal(rng, (n_slots, KW - 1, C))
    state = _normal(rng, (n_slots, Hv, D, D))
    alpha, beta = _gates(rng, (B, T, Hv), gate_form)
    z = _normal(rng, (B, T, Hv * D))
    norm_w = (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    n_keep = rng.integers(0, T + 1, size=B).astype(np.int32)
    return dict(B=B, T=T, C=C, Hk=Hk, Hv=Hv, act=act, slot_idx=slots, n_keep=n_keep,
                x=to_act(x, act), conv_w=to_act(conv_w, act),
                conv_state=to_act(conv_state, act), state=state,
                alpha=alpha, beta=beta, z=to_act(z, act), norm_w=norm_w)


def random_f32_rows(n_rows, C, *, seed, scale=1.0):
    """Plain N(0, scale^2) float32 rows, e.g. inputs of the standalone L2 norm."""
    rng = np.random.default_rng(seed)
    return _normal(rng, (n_rows, C), scale)
