"""CPU oracle of the Gated DeltaNet token-mixing path (TEST INFRASTRUCTURE).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. It wraps ``gdn_oracle.cpp`` (plain single-threaded
C++, compiled with g++ -O2 -ffp-contract=off) through ctypes. It shares no code
with the GPU library and never calls it.

Every routine takes ``prec`` = "f64" (the precision reference) or "f32" (the
same plain definitions evaluated in single precision).
Activation inputs may be float32 arrays or bfloat16 bit patterns (uint16);
they are widened exactly before the call. Results are returned unrounded
unless stated.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

D = 128


def build(force: bool = False) -> str:
    """Compile the oracle with g++ into oracle/liboracle.so (in-tree)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = ctypes.CDLL(_LIB)
        return _lib


def _swap_library(path):
    """Point the wrapper at another build of the oracle source (mutation tests
    build planted-mistake copies); path None restores the real oracle."""
    global _lib
    with _lock:
        _lib = None if path is None else ctypes.CDLL(path)


def _np_t(prec):
    return np.float64 if prec == "f64" else np.float32


def _c_t(prec):
    return ctypes.c_double if prec == "f64" else ctypes.c_float


def widen(a, prec="f64"):
    """Activation array -> float array of the oracle precision (exact)."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        a = (a.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return np.ascontiguousarray(a, dtype=_np_t(prec))


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _fn(name, prec):
    f = getattr(_load(), f"{name}_{prec}")
    return f


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _u8(a):
    return np.ascontiguousarray(a, dtype=np.uint8)


# --------------------------------------------------------------------- conv
def conv_fwd(x, conv_w, conv_state, slot_idx, cu_seqlens, has_init, Hk, Hv, *,
             silu=True, l2norm=True, eps=1e-6, prec="f64"):
    """Varlen causal conv (+SiLU, +q/k L2 norm). Returns (y, new conv_state).

    Rows of padding sequences (negative slot) stay zero in y.
    """
    T = _np_t(prec)
    xw = widen(x, prec)
    n_tok, C = xw.shape
    st = widen(conv_state, prec).copy()
    y = np.zeros((n_tok, C), T)
    f = _fn("oracle_conv_fwd", prec)
    f.restype = None
    f(_p(xw), ctypes.c_int64(n_tok), ctypes.c_int(Hk), ctypes.c_int(Hv), _p(widen(conv_w, prec)),
      _p(st), _p(_i32(slot_idx)), _p(_i32(cu_seqlens)), _p(_u8(has_init)),
      ctypes.c_int(len(slot_idx)), ctypes.c_int(int(silu)), ctypes.c_int(int(l2norm)),
      _c_t(prec)(eps), _p(y))
    return y, st


def l2norm(y, Hk, Hv, *, eps=1e-6, prec="f64"):
    """L2-normalise the q and k heads of post-conv rows (v copied)."""
    yw = widen(y, prec).copy()
    n_tok = yw.shape[0]
    f = _fn("oracle_l2norm", prec)
    f.restype = None
    f(_p(yw), ctypes.c_int64(n_tok), ctypes.c_int(Hk), ctypes.c_int(Hv), _c_t(prec)(eps))
    return yw


def tree_sum_sq(v, prec="f64"):
    vw = widen(v, prec)
    assert vw.shape == (D,)
    f = _fn("oracle_tree_sum_sq", prec)
    f.restype = _c_t(prec)
    return f(_p(vw))


def gated_rmsnorm(o, z, w, *, eps=1e-6, prec="f64"):
    ow, zw, ww = widen(o, prec), widen(z, prec), widen(w, prec)
    out = np.zeros(D, _np_t(prec))
    f = _fn("oracle_gated_rmsnorm", prec)
    f.restype = None
    f(_p(ow), _p(zw), _p(ww), _c_t(prec)(eps), _p(out))
    return out


def silu(v, prec="f64"):
    """SiLU y / (1 + exp(-y)) elementwise, with the library exp of the precision."""
    vw = widen(v, prec).copy()
    f = _fn("oracle_silu", prec)
    f.restype = None
    f(_p(vw), ctypes.c_int64(vw.size))
    return vw


def round_bf16(v, prec="f64"):
    """Round to bfloat16 values (nearest even), returned in the oracle type."""
    vw = widen(v, prec).copy()
    f = _fn("oracle_round_bf16", prec)
    f.restype = None
    f(_p(vw), ctypes.c_int64(vw.size))
    return vw


# --------------------------------------------------------------------- gates
def gates(a, b, prec="f64"):
    """The gate step from raw projections: (alpha, beta) = (exp(-softplus(a)),
    sigmoid(b)) elementwise, in the oracle precision."""
    aw, bw = widen(a, prec), widen(b, prec)
    assert aw.shape == bw.shape
    al, be = np.zeros(aw.shape, _np_t(prec)), np.zeros(bw.shape, _np_t(prec))
    f = _fn("oracle_gates", prec)
    f.restype = None
    f(_p(aw), _p(bw), ctypes.c_int64(aw.size), _p(al), _p(be))
    return al, be


# --------------------------------------------------------------------- recurrence
def prefill(qkv, alpha, beta, z, norm_w, state, slot_idx, cu_seqlens, has_init, Hk, Hv, *,
            q_scale=1.0, eps=1e-6, chunk=0, prec="f64", want_raw=False):
    """Recurrence over varlen sequences from post-conv activations.

    chunk == 0: token by token (the definition); chunk >= 1: chunked WY form.
    Returns (out, new state[, o_raw]); out rows of padding sequences stay 0.
    """
    T = _np_t(prec)
    q = widen(qkv, prec)
    n_tok = q.shape[0]
    st = widen(state, prec).copy()
    out = np.zeros((n_tok, Hv * D), T)
    raw = np.zeros((n_tok, Hv * D), T) if want_raw else None
    f = _fn("oracle_prefill", prec)
    f.restype = None
    f(_p(q), _p(widen(alpha, prec)), _p(widen(beta, prec)), _p(widen(z, prec)),
      _p(widen(norm_w, prec)), _p(st), _p(_i32(slot_idx)), _p(_i32(cu_seqlens)),
      _p(_u8(has_init)), ctypes.c_int(len(slot_idx)), ctypes.c_int(Hk), ctypes.c_int(Hv),
      _c_t(prec)(q_scale), _c_t(prec)(eps), ctypes.c_int(chunk), _p(out), _p(raw))
    return (out, st, raw) if want_raw else (out, st)


def verify(x, conv_w, conv_state, state, alpha, beta, z, norm_w, slot_idx, Hk, Hv, *,
           q_scale=1.0, eps=1e-6, round_act=False, commit_all=False, prec="f64",
           want_raw=False):
    """Speculative verify of T draft tokens (x [B][T][C]).

    round_act: round the post-conv activations to bfloat16 before the
    recurrence (activations that went through memory). The fused verify,
    commit and decode kernels keep them on chip unrounded, hence the default.

    Returns (out [B][T][Hv*D], postconv [B][T][C], conv_state', state'[, o_raw]);
    the states are unchanged copies unless commit_all.
    """
    T = _np_t(prec)
    xw = widen(x, prec)
    B, Tn, C = xw.shape
    cs = widen(conv_state, prec).copy()
    st = widen(state, prec).copy()
    out = np.zeros((B, Tn, Hv * D), T)
    pc = np.zeros((B, Tn, C), T)
    raw = np.zeros((B, Tn, Hv * D), T) if want_raw else None
    f = _fn("oracle_verify", prec)
    f.restype = None
    f(_p(xw), _p(widen(conv_w, prec)), _p(cs), _p(st), _p(widen(alpha, prec)),
      _p(widen(beta, prec)), _p(widen(z, prec)), _p(widen(norm_w, prec)), _p(_i32(slot_idx)),
      ctypes.c_int(B), ctypes.c_int(Tn), ctypes.c_int(Hk), ctypes.c_int(Hv),
      _c_t(prec)(q_scale), _c_t(prec)(eps), ctypes.c_int(int(round_act)),
      ctypes.c_int(int(commit_all)), _p(out), _p(pc), _p(raw))
    return (out, pc, cs, st, raw) if want_raw else (out, pc, cs, st)


def commit(x, alpha, beta, conv_w, conv_state, state, slot_idx, n_keep, Hk, Hv, *,
           eps=1e-6, round_act=False, prec="f64"):
    """Commit the accepted prefix n_keep[b] of one layer (round_act as for
    verify). Returns (conv_state', state')."""
    xw = widen(x, prec)
    B, Tn, C = xw.shape
    cs = widen(conv_state, prec).copy()
    st = widen(state, prec).copy()
    f = _fn("oracle_commit", prec)
    f.restype = None
    f(_p(xw), _p(widen(alpha, prec)), _p(widen(beta, prec)), _p(widen(conv_w, prec)), _p(cs),
      _p(st), _p(_i32(slot_idx)), _p(_i32(n_keep)), ctypes.c_int(B), ctypes.c_int(Tn),
      ctypes.c_int(Hk), ctypes.c_int(Hv), _c_t(prec)(eps), ctypes.c_int(int(round_act)))
    return cs, st
