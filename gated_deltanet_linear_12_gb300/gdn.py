"""ctypes binding of libgdn.so: the C ABI of include/gdn.h with the same names.

Argument marshalling only — every step of the path runs in the library's CUDA
kernels. Tensors are PyTorch CUDA tensors (device memory); the current torch
stream of the tensors' device is passed unless a stream is given. A non-OK
status raises GdnError. If libgdn.so is missing the first call raises: there is
no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

GDN_OK, GDN_ERR_INVALID, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA = 0, 1, 2, 3
GDN_F32, GDN_BF16 = 0, 1
GDN_VERIFY_COMMIT_ALL = 1
GDN_GATES_ACTIVATED, GDN_GATES_RAW = 0, 1
GDN_DEVERR_SLOT, GDN_DEVERR_NKEEP, GDN_DEVERR_SEQLENS, GDN_DEVERR_TIMEOUT = 1, 2, 4, 8
HEAD_DIM, CONV_WIDTH, CHUNK, MAX_DRAFT = 128, 4, 64, 8

EXPORTS = ["gdn_conv_fwd", "gdn_postconv_norm", "gdn_delta_prefill", "gdn_verify_workspace_bytes",
           "gdn_verify_step", "gdn_verify_step_noalloc",
           "gdn_commit_layers", "gdn_gates", "gdn_verify_step_lazy", "gdn_selftest_tc_gemm", "gdn_selftest_tc_gemm_tf32", "gdn_status_string"]


class GdnError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn} returned {status} ({msg})")
        self.status = status


class GdnConfig(ctypes.Structure):
    _fields_ = [("n_qk_heads", ctypes.c_int32), ("n_v_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("conv_width", ctypes.c_int32),
                ("act", ctypes.c_int32), ("eps", ctypes.c_float), ("q_scale", ctypes.c_float),
                ("n_slots", ctypes.c_int32), ("dev_err", ctypes.c_void_p), ("gates", ctypes.c_int32),
                ("gate_dtype", ctypes.c_int32), ("out_f32", ctypes.c_int32)]


class GdnLayerView(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("alpha", ctypes.c_void_p), ("beta", ctypes.c_void_p),
                ("conv_w", ctypes.c_void_p), ("conv_state", ctypes.c_void_p),
                ("state", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libgdn.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise RuntimeError(f"{_build.LIB} is missing: build it with "
                                   "gated_deltanet_linear_12_gb300.build.build()")
            L = ctypes.CDLL(_build.LIB)
            vp, i32, i64, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
            cfgp = ctypes.POINTER(GdnConfig)
            L.gdn_conv_fwd.argtypes = [cfgp, vp, i64, vp, i64, vp, vp, vp, vp, vp, i32, i64, i32, vp]
            L.gdn_postconv_norm.argtypes = [cfgp, i32, vp, i32, vp, i64, vp]
            L.gdn_delta_prefill.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i64,
                                            i32, vp]
            L.gdn_verify_workspace_bytes.argtypes = [cfgp, i32, i32]
            L.gdn_verify_step.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                          u32, vp, vp, i64, vp]
            L.gdn_verify_step_noalloc.argtypes = [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                                  i32, vp, vp]
            L.gdn_commit_layers.argtypes = [cfgp, vp, i32, vp, vp, i32, i32, vp]
            L.gdn_gates.argtypes = [cfgp, vp, vp, vp, vp, i64, vp]
            L.gdn_verify_step_lazy.argtypes = [cfgp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp,
                                               vp, vp, vp, i32, i32, vp, vp]
            L.gdn_selftest_tc_gemm.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp]
            L.gdn_selftest_tc_gemm_tf32.argtypes = [vp, vp, vp, i32, i32, vp, vp]
            for f in EXPORTS[:-1]:
                getattr(L, f).restype = ctypes.c_int
            L.gdn_verify_workspace_bytes.restype = ctypes.c_int64
            L.gdn_status_string.argtypes = [ctypes.c_int]
            L.gdn_status_string.restype = ctypes.c_char_p
            _lib = L
        return _lib


def status_string(status: int) -> str:
    return load().gdn_status_string(status).decode()


def _check(fn, status):
    if status != GDN_OK:
        raise GdnError(fn, status, status_string(status))


def act_of(dtype: torch.dtype) -> int:
    if dtype == torch.bfloat16:
        return GDN_BF16
    if dtype == torch.float32:
        return GDN_F32
    raise ValueError(f"unsupported activation dtype {dtype}")


def make_config(n_qk_heads, n_v_heads, act, n_slots, *, eps=1e-6, q_scale=1.0, dev_err=None,
                gates=GDN_GATES_ACTIVATED, gate_dtype=GDN_F32, out_f32=False):
    """gdn_config; act and gate_dtype are GDN_F32/GDN_BF16 or torch dtypes; dev_err a
    CUDA int32 tensor; gates GDN_GATES_RAW makes alpha / beta arguments raw
    projections; out_f32 makes `out` f32 whatever the activation dtype."""
    if isinstance(act, torch.dtype):
        act = act_of(act)
    if isinstance(gate_dtype, torch.dtype):
        gate_dtype = act_of(gate_dtype)
    return GdnConfig(n_qk_heads, n_v_heads, HEAD_DIM, CONV_WIDTH, act, eps, q_scale, n_slots,
                     dev_err.data_ptr() if dev_err is not None else None, gates, gate_dtype,
                     int(bool(out_f32)))


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    return t.data_ptr()


def _stream(t, stream):
    if stream is not None:
        return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)
    return torch.cuda.current_stream(t.device).cuda_stream


def _dense(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensor must be contiguous")


# ----------------------------------------------------------------------------- entry points
def gdn_conv_fwd(cfg, x, y, conv_w, conv_state, slot_idx, cu_seqlens, has_init, *,
                 fuse_norm=True, stream=None):
    """x, y: [n_tok][>=C] (row stride = leading dimension); see include/gdn.h."""
    if x.stride(1) != 1 or y.stride(1) != 1:
        raise ValueError("x and y rows must be contiguous")
    _dense(conv_w, conv_state, slot_idx, cu_seqlens, has_init)
    _check("gdn_conv_fwd", load().gdn_conv_fwd(
        ctypes.byref(cfg), _ptr(x), x.stride(0), _ptr(y), y.stride(0), _ptr(conv_w),
        _ptr(conv_state), _ptr(slot_idx), _ptr(cu_seqlens), _ptr(has_init), slot_idx.numel(),
        x.shape[0], int(bool(fuse_norm)), _stream(x, stream)))


def gdn_postconv_norm(cfg, y_in, y_out, *, stream=None):
    _dense(y_in, y_out)
    _check("gdn_postconv_norm", load().gdn_postconv_norm(
        ctypes.byref(cfg), act_of(y_in.dtype), _ptr(y_in), act_of(y_out.dtype), _ptr(y_out),
        y_in.shape[0], _stream(y_in, stream)))


def gdn_delta_prefill(cfg, qkv, alpha, beta, z, norm_w, out, state, slot_idx, cu_seqlens,
                      has_init, *, chunk=CHUNK, stream=None):
    _dense(qkv, alpha, beta, z, norm_w, out, state, slot_idx, cu_seqlens, has_init)
    _check("gdn_delta_prefill", load().gdn_delta_prefill(
        ctypes.byref(cfg), _ptr(qkv), _ptr(alpha), _ptr(beta), _ptr(z), _ptr(norm_w), _ptr(out),
        _ptr(state), _ptr(slot_idx), _ptr(cu_seqlens), _ptr(has_init), slot_idx.numel(),
        qkv.shape[0], chunk, _stream(qkv, stream)))


def gdn_verify_workspace_bytes(cfg, B, T):
    n = load().gdn_verify_workspace_bytes(ctypes.byref(cfg), B, T)
    if n < 0:
        raise GdnError("gdn_verify_workspace_bytes", GDN_ERR_INVALID, "invalid configuration")
    return n


def verify_workspace(cfg, B, T, device):
    """A device buffer for gdn_verify_step's workspace argument, or None when the
    configuration needs none (the current kernel needs none)."""
    n = gdn_verify_workspace_bytes(cfg, B, T)
    return torch.zeros(n, dtype=torch.uint8, device=device) if n > 0 else None


def gdn_verify_step(cfg, x, conv_w, conv_state, state, alpha, beta, z, norm_w, out, slot_idx, *,
                    commit_all=False, postconv_out=None, workspace=None, stream=None):
    """x [B][T][C]; alpha, beta [B][T][Hv]; z, out [B][T][Hv*128]. workspace: a
    uint8 CUDA tensor from verify_workspace, or None (sized by the library when
    omitted; the current kernel needs none)."""
    _dense(x, conv_w, conv_state, state, alpha, beta, z, norm_w, out, slot_idx, postconv_out)
    B, T = x.shape[0], x.shape[1]
    ws, ws_bytes = None, 0
    if not commit_all:
        if workspace is None:
            workspace = verify_workspace(cfg, B, T, x.device)
        if workspace is not None:
            _dense(workspace)
            ws, ws_bytes = workspace, workspace.numel() * workspace.element_size()
    _check("gdn_verify_step", load().gdn_verify_step(
        ctypes.byref(cfg), _ptr(x), _ptr(conv_w), _ptr(conv_state), _ptr(state), _ptr(alpha),
        _ptr(beta), _ptr(z), _ptr(norm_w), _ptr(out), _ptr(slot_idx), B, T,
        GDN_VERIFY_COMMIT_ALL if commit_all else 0, _ptr(postconv_out), _ptr(ws), ws_bytes,
        _stream(x, stream)))


def make_layer_views(layers, device):
    """Device array [L] of gdn_layer_view from dicts with keys x, alpha, beta,
    conv_w, conv_state, state (CUDA tensors). Returns a uint8 CUDA tensor; the
    tensors it points to must outlive its use."""
    arr = (GdnLayerView * len(layers))()
    for i, l in enumerate(layers):
        arr[i] = GdnLayerView(_ptr(l["x"]), _ptr(l["alpha"]), _ptr(l["beta"]), _ptr(l["conv_w"]),
                              _ptr(l["conv_state"]), _ptr(l["state"]))
    raw = bytes(arr)
    host = torch.frombuffer(bytearray(raw), dtype=torch.uint8)
    return host.to(device)


def gdn_verify_step_noalloc(cfg, x, conv_w, conv_state, state, alpha, beta, z, norm_w, out, slot_idx, *,
                            postconv_out=None, stream=None):
    """Read-only verify that allocates nothing and takes no workspace: it
    launches the same kernel as gdn_verify_step. Same arrays as gdn_verify_step."""
    _dense(x, conv_w, conv_state, state, alpha, beta, z, norm_w, out, slot_idx, postconv_out)
    B, T = x.shape[0], x.shape[1]
    _check("gdn_verify_step_noalloc", load().gdn_verify_step_noalloc(
        ctypes.byref(cfg), _ptr(x), _ptr(conv_w), _ptr(conv_state), _ptr(state), _ptr(alpha),
        _ptr(beta), _ptr(z), _ptr(norm_w), _ptr(out), _ptr(slot_idx), B, T, _ptr(postconv_out),
        _stream(x, stream)))


def gdn_commit_layers(cfg, views, n_layers, slot_idx, n_keep, T, *, stream=None):
    """views: uint8 CUDA tensor from make_layer_views (n_layers entries)."""
    _dense(slot_idx, n_keep)
    _check("gdn_commit_layers", load().gdn_commit_layers(
        ctypes.byref(cfg), _ptr(views), n_layers, _ptr(slot_idx), _ptr(n_keep), slot_idx.numel(),
        T, _stream(slot_idx, stream)))


def gdn_verify_step_lazy(cfg, prev_x, prev_alpha, prev_beta, prev_n_keep, x, conv_w, conv_state,
                         state, alpha, beta, z, norm_w, out, slot_idx, *, postconv_out=None,
                         stream=None):
    """Verify of x's T drafts with the previous window's accepted prefixes
    (prev_x [B][prev_T][C], prev_n_keep [B]) committed first, in one launch."""
    _dense(prev_x, prev_alpha, prev_beta, prev_n_keep, x, conv_w, conv_state, state, alpha, beta,
           z, norm_w, out, slot_idx, postconv_out)
    B, T = x.shape[0], x.shape[1]
    if prev_x.shape[0] != B:
        raise ValueError("prev_x and x must have the same batch")
    _check("gdn_verify_step_lazy", load().gdn_verify_step_lazy(
        ctypes.byref(cfg), _ptr(prev_x), _ptr(prev_alpha), _ptr(prev_beta), _ptr(prev_n_keep),
        prev_x.shape[1], _ptr(x), _ptr(conv_w), _ptr(conv_state), _ptr(state), _ptr(alpha),
        _ptr(beta), _ptr(z), _ptr(norm_w), _ptr(out), _ptr(slot_idx), B, T, _ptr(postconv_out),
        _stream(x, stream)))


def gdn_gates(cfg, a, b, alpha, beta, *, stream=None):
    """alpha = exp(-softplus(a)), beta = sigmoid(b) for tensors of the same shape
    whose last dimension is Hv ([n_tok][Hv] or [B][T][Hv]), of the config's
    gate dtype (float32 or bfloat16)."""
    _dense(a, b, alpha, beta)
    if not (a.shape == b.shape == alpha.shape == beta.shape) or a.shape[-1] != cfg.n_v_heads:
        raise ValueError("a, b, alpha, beta must share one shape [..., Hv]")
    want = torch.bfloat16 if cfg.gate_dtype == GDN_BF16 else torch.float32
    if any(t.dtype != want for t in (a, b, alpha, beta)):
        raise ValueError(f"gates must be {want} (the config's gate_dtype)")
    _check("gdn_gates", load().gdn_gates(ctypes.byref(cfg), _ptr(a), _ptr(b), _ptr(alpha), _ptr(beta),
                                         a.numel() // cfg.n_v_heads, _stream(a, stream)))


def gdn_selftest_tc_gemm(A, B, D, *, starve_wait=False, dev_err=None, stream=None):
    """Diagnostic: D[128][N] = A[128][K] @ B[N][K]^T on the tensor cores (bf16 -> f32).
    starve_wait exercises the bounded-wait failure path (see gdn_selftest.h)."""
    _dense(A, B, D)
    _check("gdn_selftest_tc_gemm", load().gdn_selftest_tc_gemm(
        _ptr(A), _ptr(B), _ptr(D), B.shape[0], A.shape[1], int(bool(starve_wait)),
        _ptr(dev_err), _stream(A, stream)))


def gdn_selftest_tc_gemm_tf32(A, B, D, *, dev_err=None, stream=None):
    """Diagnostic: D[128][N] = A[128][K] @ B[N][K]^T, f32 operands on the tf32 path."""
    _dense(A, B, D)
    _check("gdn_selftest_tc_gemm_tf32", load().gdn_selftest_tc_gemm_tf32(
        _ptr(A), _ptr(B), _ptr(D), B.shape[0], A.shape[1], _ptr(dev_err), _stream(A, stream)))
