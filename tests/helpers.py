"""Shared helpers of the tests: tensor transfer and the tolerance checks.

Tolerances (floating point; integer, index and state-commit results are bitwise):
  f32 conv / norm outputs   |gpu - ref| <= 1e-5 * max(|ref|, 1e-30) against the
                            oracle's float instantiation (the same tap-ordered
                            sum, so equal pre-activations), and
                            |gpu - ref| <= 1e-5 * max(|ref|, kappa) against the
                            double one, kappa = 1.1 r sum_j |w_j x_j| (the scale
                            the f32 conv sum is accurate to; r the head's L2
                            factor, 1 for v heads)
  f32 recurrence outputs    |gpu - ref| <= 1e-4 * max(1, |ref|)
  bf16 outputs              |gpu - ref| <= max(2e-2, 1 bf16 ulp of ref), ref unrounded
  f32 recurrent states      ||gpu - ref||_F <= 1e-4 ||ref||_F per (slot, head)
"""
import math

import numpy as np

D = 128


def to_dev(a, act=None, device="cuda"):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def to_np(t):
    """CUDA tensor -> numpy float64 (bf16 widened exactly)."""
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.float().numpy().astype(np.float64)
    return t.numpy().astype(np.float64)


def bits(t):
    """Raw bit patterns of a CUDA tensor as a numpy array (for bitwise checks)."""
    import torch
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy()
    return t.numpy()


class Canary:
    """Copies of device tensors placed between guard bands of a NaN bit pattern
    (512 bytes on each side, so alignment is kept): check() asserts that no
    kernel wrote outside the tensors it was given."""

    PATTERN = {2: 0x7FD1, 4: 0x7FC0DEAD}           # quiet NaNs of bf16 and f32

    def __init__(self):
        self.guards = []

    def wrap(self, t):
        import torch
        es = t.element_size()
        band = 512 // es
        n = t.numel()
        raw = torch.empty(n + 2 * band, dtype=t.dtype, device=t.device)
        iview = raw.view(torch.int16 if es == 2 else torch.int32)
        pat = self.PATTERN[es]
        iview.fill_(pat - (1 << 16) if es == 2 and pat >= 1 << 15 else pat)
        inner = raw[band:band + n].view(t.shape)
        inner.copy_(t)
        self.guards.append((raw, band, n, pat, es))
        return inner

    def check(self, what=""):
        for raw, band, n, pat, es in self.guards:
            b = bits(raw).astype(np.int64) & ((1 << (8 * es)) - 1)
            assert np.all(b[:band] == pat) and np.all(b[band + n:] == pat), (
                f"{what}: a kernel wrote into the guard band of a {tuple(raw.shape)} buffer")


def bf16_ulp(ref):
    a = np.abs(np.asarray(ref, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def check_bf16(gpu, ref, atol=2e-2, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref)
    bound = np.maximum(atol, bf16_ulp(ref))
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} bf16 elements out of tolerance; "
                           f"max err {err.max():.3g}")
    return int((err > atol).sum())      # count above 2e-2 (allowed by the 1-ulp reading)


def check_f32_rel(gpu, ref, rtol=1e-5, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref) / np.maximum(np.abs(ref), 1e-30)
    assert err.max() <= rtol, f"{what}: max relative error {err.max():.3g} > {rtol}"


def conv_kappa(orc, x, conv_w, conv_state, slot_idx, cu_seqlens, has_init, Hk, Hv, eps=1e-6,
               l2norm=True):
    """kappa of the f32 conv/norm tolerance against the double oracle, per element."""
    ab = lambda a: np.abs(orc.widen(a))
    A, _ = orc.conv_fwd(ab(x), ab(conv_w), ab(conv_state), slot_idx, cu_seqlens, has_init, Hk, Hv,
                        silu=False, l2norm=False)
    s, _ = orc.conv_fwd(x, conv_w, conv_state, slot_idx, cu_seqlens, has_init, Hk, Hv,
                        l2norm=False)
    n, C = s.shape
    heads = s.reshape(n, C // D, D)
    r = 1.0 / np.sqrt((heads * heads).sum(axis=2, keepdims=True) + eps)
    r[:, 2 * Hk:] = 1.0                                   # v heads are not normalised
    if not l2norm:
        r[:] = 1.0
    return 1.1 * A * np.broadcast_to(r, heads.shape).reshape(n, C)


def check_f32_cond(gpu, ref, kappa, rtol=1e-5, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref) / np.maximum(np.maximum(np.abs(ref), kappa), 1e-30)
    assert err.max() <= rtol, f"{what}: max conditioned relative error {err.max():.3g} > {rtol}"


def check_f32_out(gpu, ref, tol=1e-4, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref) / np.maximum(1.0, np.abs(ref))
    assert err.max() <= tol, f"{what}: max scaled error {err.max():.3g} > {tol}"


def check_states(gpu, ref, slots, tol=1e-4, what=""):
    """Relative Frobenius error per (slot, head) of [n_slots][Hv][D][D] pools."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    worst = 0.0
    for s in slots:
        for h in range(ref.shape[1]):
            n = np.linalg.norm(ref[s, h])
            e = np.linalg.norm(gpu[s, h] - ref[s, h])
            r = e / n if n > 0 else e
            worst = max(worst, r)
            assert r <= tol, f"{what}: slot {s} head {h} relative Frobenius error {r:.3g} > {tol}"
    return worst
