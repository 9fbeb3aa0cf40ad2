"""CPU checks of the C ABI: the library builds for sm_103a, exports every entry
point include/gdn.h declares, and rejects bad arguments on the host before any
CUDA call (so these run without a GPU: no compute call is made)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", h) for h in sorted(os.listdir(os.path.join(ROOT, "include")))
           if h.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    from gated_deltanet_linear_12_gb300 import build, gdn
    build.build()
    return gdn.load()


def declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    return sorted(set(re.findall(r"^\s*(?:gdn_status|const char\*)\s+(gdn_\w+)\s*\(", text, re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 7
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings(lib):
    from gated_deltanet_linear_12_gb300 import gdn
    assert gdn.status_string(0) == "ok"
    assert "invalid" in gdn.status_string(1)
    assert "unsupported" in gdn.status_string(2)


def _cfg(**kw):
    from gated_deltanet_linear_12_gb300 import gdn
    c = gdn.GdnConfig(2, 4, 128, 4, gdn.GDN_BF16, 1e-6, 1.0, 8, None)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


# Fake, 16-byte aligned device addresses: validation rejects before any use.
P = [0x7f0000000000 + i * 0x10000000 for i in range(16)]


def _conv(lib, cfg, x=P[0], ldx=1024, y=P[1], ldy=1024, n_seq=2, n_tok=100):
    return lib.gdn_conv_fwd(ctypes.byref(cfg) if cfg is not None else None, x, ldx, y, ldy, P[2],
                            P[3], P[4], P[5], P[6], n_seq, n_tok, 1, None)


def test_conv_host_validation(lib):
    assert _conv(lib, None) == 1
    assert _conv(lib, _cfg(head_dim=64)) == 2
    assert _conv(lib, _cfg(conv_width=3)) == 2
    assert _conv(lib, _cfg(act=7)) == 2
    assert _conv(lib, _cfg(n_v_heads=3)) == 1            # Hv % Hk != 0
    assert _conv(lib, _cfg(n_qk_heads=1, n_v_heads=17)) == 2   # group too large
    assert _conv(lib, _cfg(n_slots=0)) == 1
    assert _conv(lib, _cfg(), x=0) == 1
    assert _conv(lib, _cfg(), y=P[0]) == 1               # y overlaps x
    assert _conv(lib, _cfg(), x=P[0] + 8) == 1           # misaligned
    assert _conv(lib, _cfg(), ldx=1000) == 1             # ld < C
    assert _conv(lib, _cfg(), ldx=1028) == 1             # row not 16-byte aligned
    assert _conv(lib, _cfg(), n_seq=-1) == 1
    assert _conv(lib, _cfg(), n_seq=0) == 0              # empty batch: no-op


def test_postconv_norm_host_validation(lib):
    c = _cfg()
    assert lib.gdn_postconv_norm(ctypes.byref(c), 3, P[0], 1, P[1], 10, None) == 2
    assert lib.gdn_postconv_norm(ctypes.byref(c), 1, P[0], 1, P[0] + 64, 10, None) == 1
    assert lib.gdn_postconv_norm(ctypes.byref(c), 1, P[0], 1, P[1], 0, None) == 0
    assert lib.gdn_postconv_norm(ctypes.byref(c), 1, 0, 1, P[1], 5, None) == 1


def test_prefill_host_validation(lib):
    c = _cfg()
    args = [P[i] for i in range(10)]
    assert lib.gdn_delta_prefill(ctypes.byref(c), *args, 2, 100, 32, None) == 2   # chunk
    assert lib.gdn_delta_prefill(ctypes.byref(c), *args, 0, 100, 64, None) == 0
    bad = list(args)
    bad[5] = P[0]                                          # out aliases qkv
    assert lib.gdn_delta_prefill(ctypes.byref(c), *bad, 2, 100, 64, None) == 1
    bad = list(args)
    bad[6] = 0                                             # state null
    assert lib.gdn_delta_prefill(ctypes.byref(c), *bad, 2, 100, 64, None) == 1


def test_verify_and_commit_host_validation(lib):
    c = _cfg()
    v = [P[i] for i in range(10)]
    ws = P[10]
    assert lib.gdn_verify_workspace_bytes(ctypes.byref(c), 4, 2) == 0       # the kernel needs none
    assert lib.gdn_verify_workspace_bytes(ctypes.byref(c), 4, 9) == -1
    assert lib.gdn_verify_step(ctypes.byref(c), *v, 4, 9, 0, None, None, 0, None) == 1   # T > 8
    assert lib.gdn_verify_step(ctypes.byref(c), *v, 4, 0, 0, None, None, 0, None) == 1   # T < 1
    assert lib.gdn_verify_step(ctypes.byref(c), *v, 4, 2, 4, None, None, 0, None) == 1   # bad flag
    assert lib.gdn_verify_step(ctypes.byref(c), *v, 0, 2, 0, None, None, 0, None) == 0   # B = 0
    assert lib.gdn_verify_step(ctypes.byref(c), *v, 4, 2, 0, None, ws, -1, None) == 1    # negative size
    assert lib.gdn_verify_step(ctypes.byref(c), *v, 4, 2, 0, None, None, 256, None) == 1  # NULL, size != 0
    assert lib.gdn_verify_step_noalloc(ctypes.byref(c), *v, 4, 9, None, None) == 1       # T > 8
    assert lib.gdn_verify_step_noalloc(ctypes.byref(c), *v, 0, 2, None, None) == 0       # B = 0
    assert lib.gdn_commit_layers(ctypes.byref(c), P[0], 36, P[1], P[2], 4, 0, None) == 1
    assert lib.gdn_commit_layers(ctypes.byref(c), 0, 36, P[1], P[2], 4, 2, None) == 1
    assert lib.gdn_commit_layers(ctypes.byref(c), P[0], 0, P[1], P[2], 4, 2, None) == 0


def test_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    from gated_deltanet_linear_12_gb300 import gdn
    cfg = gdn.make_config(1, 1, torch.float32, 1)
    t = torch.zeros(4, 384)
    with pytest.raises(ValueError):
        gdn.gdn_postconv_norm(cfg, t, t)


def test_gates_mode_and_gdn_gates_host_validation(lib):
    """An unknown gates mode is rejected by every entry that reads the config;
    gdn_gates rejects null pointers, negative sizes and overlaps other than in
    place, and enqueues nothing for n_tok = 0."""
    assert _conv(lib, _cfg(gates=2)) == 1
    assert _conv(lib, _cfg(gates=-1)) == 1
    c = _cfg()
    c_raw = _cfg(gates=1)
    n = 10
    nb = n * 4 * 4                                          # n_tok x Hv f32
    assert lib.gdn_gates(None, P[0], P[1], P[2], P[3], n, None) == 1
    assert lib.gdn_gates(ctypes.byref(c), P[0], P[1], P[2], P[3], -1, None) == 1
    assert lib.gdn_gates(ctypes.byref(c), P[0], P[1], P[2], P[3], 0, None) == 0
    assert lib.gdn_gates(ctypes.byref(c_raw), 0, 0, 0, 0, 0, None) == 0
    assert lib.gdn_gates(ctypes.byref(c), 0, P[1], P[2], P[3], n, None) == 1
    assert lib.gdn_gates(ctypes.byref(c), P[0], P[1], P[2], 0, n, None) == 1
    assert lib.gdn_gates(ctypes.byref(c), P[0], P[1], P[2], P[2] + nb - 4, n, None) == 1   # alpha/beta
    assert lib.gdn_gates(ctypes.byref(c), P[0], P[1], P[1], P[3], n, None) == 1            # alpha = b
    assert lib.gdn_gates(ctypes.byref(c), P[0], P[1], P[0] + 4, P[3], n, None) == 1        # shifted a
    assert lib.gdn_gates(ctypes.byref(c), P[0], P[1], P[2], P[0], n, None) == 1            # beta = a


def test_verify_lazy_host_validation(lib):
    c = _cfg()
    prev = [P[11], P[12], P[13], P[14]]                     # prev_x, prev_alpha, prev_beta, n_keep
    v = [P[i] for i in range(10)]

    def call(prev_args, prev_T, B, T, vv=v, post=None, cfg=c):
        return lib.gdn_verify_step_lazy(ctypes.byref(cfg), *prev_args, prev_T, *vv, B, T, post, None)

    assert call(prev, 4, 0, 2) == 0                          # B = 0 enqueues nothing
    assert call(prev, 4, 4, 9) == 1                          # T > 8
    assert call(prev, 0, 4, 2) == 1                          # prev_T < 1
    assert call(prev, 9, 4, 2) == 1                          # prev_T > 8
    assert call([0] + prev[1:], 4, 4, 2) == 1                # null prev_x
    assert call(prev[:3] + [0], 4, 4, 2) == 1                # null prev_n_keep
    assert call([P[11] + 8] + prev[1:], 4, 4, 2) == 1        # misaligned prev_x
    bad = list(v)
    bad[8] = P[11]                                           # out = prev_x
    assert call(prev, 4, 4, 2, vv=bad) == 1
    assert call(prev, 4, 4, 2, post=P[15] + 4) == 1          # misaligned post-conv output
    assert call(prev, 4, 4, 2, cfg=_cfg(gates=3)) == 1


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    """No fallback: with libgdn.so absent the binding raises instead of computing
    anything another way."""
    from gated_deltanet_linear_12_gb300 import build, gdn
    monkeypatch.setattr(build, "LIB", str(tmp_path / "libgdn.so"))
    monkeypatch.setattr(gdn, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        gdn.load()


def test_build_compiles_every_cuda_source():
    """Every translation unit under csrc/ is in the build, and every header it lists exists."""
    from gated_deltanet_linear_12_gb300 import build
    cu = sorted(f for f in os.listdir(build.CSRC) if f.endswith(".cu"))
    assert sorted(build.SOURCES) == cu
    hdr = sorted(f for f in os.listdir(build.CSRC) if f.endswith((".cuh", ".h")))
    assert sorted(build.HEADERS) == hdr                # an edited header triggers a rebuild
