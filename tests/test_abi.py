"""The C-ABI library builds for sm_103a, loads, exports every function that
include/qkvp.h declares, and validates arguments on the host before touching
the GPU.  CPU only: no call here reaches a kernel launch."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qkvp.h")


@pytest.fixture(scope="module")
def qk():
    from fp8_packed_reduced_gb300 import build as b
    try:
        b.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    b.build()
    import fp8_packed_reduced_gb300 as pkg
    pkg.lib()
    return pkg


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(qkvp_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


def test_header_declares_the_calls():
    names = _declared_functions()
    for n in ("qkvp_quantize_bank", "qkvp_forward", "qkvp_backward", "qkvp_workspace_bytes",
              "qkvp_build_rope_table", "qkvp_poll_device_status", "qkvp_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(qk):
    L = ctypes.CDLL(qk.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_status_strings(qk):
    for code, name in qk.STATUS.items():
        assert qk.lib().qkvp_status_string(code).decode() == name
    assert qk.lib().qkvp_status_string(99).decode() == "QKVP_ERR_UNKNOWN"


def test_workspace_sizes(qk):
    assert qk.workspace_bytes(qk.Shape(128, 768, 6)) > 0
    assert qk.workspace_bytes(qk.Shape(128, 768, 6, d_qk=80)) == 0      # unsupported width
    assert qk.workspace_bytes(qk.Shape(128, 700, 6)) == 0               # D not a multiple of 128
    assert qk.lib().qkvp_bank_workspace_bytes(12, 768, 6, 96, 128) > 0
    assert qk.lib().qkvp_bank_workspace_bytes(0, 768, 6, 96, 128) == 0


def _fwd(qk, dims, ws_bytes=1 << 40, eps=1e-6, max_pos=128, ptr=4096, null_at=None):
    # args[0] is the rope table, args[1:] the 11 tensor pointers x .. ws, in order
    args = [ctypes.c_void_p(ptr) for _ in range(12)]
    if null_at is not None:
        args[null_at] = None
    return qk.lib().qkvp_forward(ctypes.byref(dims), eps, args[0], max_pos, *args[1:], ws_bytes, None)


def test_forward_validation_codes(qk):
    good = qk.Dims(128, 768, 6, 96, 128)
    assert _fwd(qk, qk.Dims(0, 768, 6, 96, 128)) == qk.ERR_INVALID_ARGUMENT
    assert _fwd(qk, qk.Dims(128, 768, 6, 80, 128)) == qk.ERR_UNSUPPORTED
    assert _fwd(qk, qk.Dims(128, 768, 6, 96, 64)) == qk.ERR_UNSUPPORTED
    assert _fwd(qk, qk.Dims(128, 640 + 64, 6, 96, 128)) == qk.ERR_UNSUPPORTED
    assert _fwd(qk, good, null_at=3) == qk.ERR_INVALID_ARGUMENT
    assert _fwd(qk, good, max_pos=0) == qk.ERR_INVALID_ARGUMENT
    assert _fwd(qk, good, eps=-1.0) == qk.ERR_INVALID_ARGUMENT
    assert _fwd(qk, good, ptr=4104) == qk.ERR_MISALIGNED
    assert _fwd(qk, good, ws_bytes=16) == qk.ERR_WORKSPACE_TOO_SMALL


def test_backward_validation_codes(qk):
    good = qk.Dims(200, 1024, 8, 128, 128)
    # P[0] is the rope table, P[1:] the 16 tensor pointers dq .. ws, in order
    P = [ctypes.c_void_p(8192) for _ in range(17)]
    call = lambda dims, P, ws=1 << 40: qk.lib().qkvp_backward(ctypes.byref(dims), P[0], 64, *P[1:], ws, None)
    assert call(qk.Dims(200, 1024, 8, 100, 128), P) == qk.ERR_UNSUPPORTED
    bad = list(P)
    bad[5] = None
    assert call(good, bad) == qk.ERR_INVALID_ARGUMENT
    bad = list(P)
    bad[7] = ctypes.c_void_p(8200)
    assert call(good, bad) == qk.ERR_MISALIGNED
    assert call(good, P, ws=100) == qk.ERR_WORKSPACE_TOO_SMALL


def test_bank_validation_codes(qk):
    L = 2
    arr = (ctypes.c_void_p * L)(ctypes.c_void_p(4096), ctypes.c_void_p(4096))
    p = ctypes.c_void_p(4096)
    f = qk.lib().qkvp_quantize_bank
    assert f(0, 768, 6, 96, 128, arr, arr, arr, p, p, p, p, 1 << 20, None) == qk.ERR_INVALID_ARGUMENT
    assert f(L, 768, 6, 72, 128, arr, arr, arr, p, p, p, p, 1 << 20, None) == qk.ERR_UNSUPPORTED
    assert f(200, 768, 6, 96, 128, arr, arr, arr, p, p, p, p, 1 << 20, None) in (qk.ERR_UNSUPPORTED,
                                                                                 qk.ERR_INVALID_ARGUMENT)
    mis = (ctypes.c_void_p * L)(ctypes.c_void_p(4096), ctypes.c_void_p(4098))
    assert f(L, 768, 6, 96, 128, arr, mis, arr, p, p, p, p, 1 << 20, None) == qk.ERR_MISALIGNED
    assert f(L, 768, 6, 96, 128, arr, arr, arr, p, p, p, p, 8, None) == qk.ERR_WORKSPACE_TOO_SMALL


def test_static_bank_refresh_validates_like_the_workspace_one(qk):
    """The allocation-free bank refresh rejects bad arguments with the same
    status as qkvp_quantize_bank (both run the same host checks, before any
    CUDA call)."""
    L = 2
    arr = (ctypes.c_void_p * L)(ctypes.c_void_p(4096), ctypes.c_void_p(4096))
    mis = (ctypes.c_void_p * L)(ctypes.c_void_p(4096), ctypes.c_void_p(4098))
    p = ctypes.c_void_p(4096)
    lib = qk.lib()
    bad = [
        (0, 768, 6, 96, 128, arr),       # no layers
        (L, 768, 6, 72, 128, arr),       # unsupported d_qk
        (L, 768, 6, 0, 128, arr),        # non-positive d_qk
        (L, 768, 6, 96, 0, arr),         # non-positive d_v
        (L, 768, 6, 96, 64, arr),        # unsupported d_v
        (L, 700, 6, 96, 128, arr),       # D not a multiple of 128
        (L, 768, 0, 96, 128, arr),       # no heads
        (L, 768, 200, 96, 128, arr),     # too many heads
        (L, 768, 6, 96, 128, mis),       # a misaligned weight
    ]
    for L_, D, H, dqk, dv, a in bad:
        ws_rc = lib.qkvp_quantize_bank(L_, D, H, dqk, dv, a, a, a, p, p, p, p, 1 << 20, None)
        st_rc = lib.qkvp_quantize_bank_static(L_, D, H, dqk, dv, a, a, a, p, p, p, None)
        assert ws_rc == st_rc != qk.OK, (L_, D, H, dqk, dv)


def test_other_validation_codes(qk):
    lib = qk.lib()
    assert lib.qkvp_build_rope_table(None, 128, 96, 10000.0, None) == qk.ERR_INVALID_ARGUMENT
    assert lib.qkvp_build_rope_table(ctypes.c_void_p(4096), 128, 90, 10000.0, None) == qk.ERR_UNSUPPORTED
    assert lib.qkvp_build_rope_table(ctypes.c_void_p(4100), 128, 96, 10000.0, None) == qk.ERR_MISALIGNED
    assert lib.qkvp_selftest_wait_timeout(None, 256, 100, None) == qk.ERR_INVALID_ARGUMENT
    assert lib.qkvp_selftest_wait_timeout(ctypes.c_void_p(4096), 256, 0, None) == qk.ERR_INVALID_ARGUMENT
    assert lib.qkvp_set_wait_timeout_ns(10) == qk.ERR_INVALID_ARGUMENT
    assert lib.qkvp_set_wait_timeout_ns(2_000_000_000) == qk.OK
    assert lib.qkvp_workspace_init(None, 256, None) == qk.ERR_INVALID_ARGUMENT
    prev = lib.qkvp_set_cta_pairs(3)
    assert 0 <= prev <= 7
    assert lib.qkvp_set_cta_pairs(8) == -1 and lib.qkvp_set_cta_pairs(-1) == -1
    assert lib.qkvp_set_cta_pairs(prev) == 3


def test_oproj_validation_codes(qk):
    lib = qk.lib()
    p = ctypes.c_void_p(4096)
    assert lib.qkvp_oproj_workspace_bytes(128, 768, 768) > 0
    assert lib.qkvp_oproj_workspace_bytes(128, 700, 768) == 0
    assert lib.qkvp_weight_workspace_bytes(1, 768, 768) > 0
    assert lib.qkvp_weight_workspace_bytes(1, 100, 768) == 0
    fwd = lib.qkvp_oproj_forward
    assert fwd(0, 768, 768, p, p, p, p, p, p, p, 1 << 40, None) == qk.ERR_INVALID_ARGUMENT
    assert fwd(128, 700, 768, p, p, p, p, p, p, p, 1 << 40, None) == qk.ERR_UNSUPPORTED
    assert fwd(128, 768, 768, None, p, p, p, p, p, p, 1 << 40, None) == qk.ERR_INVALID_ARGUMENT
    assert fwd(128, 768, 768, ctypes.c_void_p(4100), p, p, p, p, p, p, 1 << 40, None) == qk.ERR_MISALIGNED
    assert fwd(128, 768, 768, p, p, p, p, p, p, p, 64, None) == qk.ERR_WORKSPACE_TOO_SMALL
    bwd = lib.qkvp_oproj_backward
    assert bwd(128, 768, 768, p, p, p, p, p, p, p, p, None, p, 1 << 40, None) == qk.ERR_INVALID_ARGUMENT
    assert bwd(128, 768, 640 + 1, p, p, p, p, p, p, p, p, p, p, 1 << 40, None) == qk.ERR_UNSUPPORTED
    assert bwd(128, 768, 768, p, p, p, p, p, p, p, p, p, p, 64, None) == qk.ERR_WORKSPACE_TOO_SMALL
    arr = (ctypes.c_void_p * 1)(ctypes.c_void_p(4096))
    qw = lib.qkvp_quantize_weight
    assert qw(0, 768, 768, arr, p, p, p, p, 1 << 20, None) == qk.ERR_INVALID_ARGUMENT
    assert qw(1, 768, 700, arr, p, p, p, p, 1 << 20, None) == qk.ERR_UNSUPPORTED
    assert qw(1, 768, 768, (ctypes.c_void_p * 1)(ctypes.c_void_p(4098)), p, p, p, p, 1 << 20, None) \
        == qk.ERR_MISALIGNED
    assert qw(1, 768, 768, arr, p, p, p, p, 8, None) == qk.ERR_WORKSPACE_TOO_SMALL


def test_mlp_validation_codes(qk):
    lib = qk.lib()
    p = ctypes.c_void_p(4096)
    assert lib.qkvp_mlp_workspace_bytes(128, 768, 3072) > 0
    assert lib.qkvp_mlp_workspace_bytes(128, 768, 3000) == 0
    fwd = lib.qkvp_mlp_forward
    args = [p] * 11
    assert fwd(0, 768, 3072, *args, p, 1 << 40, None) == qk.ERR_INVALID_ARGUMENT
    assert fwd(128, 768, 3000, *args, p, 1 << 40, None) == qk.ERR_UNSUPPORTED
    assert fwd(128, 768, 3072, *args, None, 1 << 40, None) == qk.ERR_INVALID_ARGUMENT
    assert fwd(128, 768, 3072, ctypes.c_void_p(4104), *args[1:], p, 1 << 40, None) == qk.ERR_MISALIGNED
    assert fwd(128, 768, 3072, *args, p, 64, None) == qk.ERR_WORKSPACE_TOO_SMALL
    bwd = lib.qkvp_mlp_backward
    bargs = [p] * 17
    assert bwd(128, 700, 3072, *bargs, p, 1 << 40, None) == qk.ERR_UNSUPPORTED
    assert bwd(128, 768, 3072, *bargs, None, 1 << 40, None) == qk.ERR_INVALID_ARGUMENT
    assert bwd(128, 768, 3072, *bargs, p, 64, None) == qk.ERR_WORKSPACE_TOO_SMALL


def test_split_forward_validation_codes(qk):
    lib = qk.lib()
    p = ctypes.c_void_p(4096)
    n = lib.qkvp_activation_workspace_bytes()
    assert n > 0
    qa = lib.qkvp_quantize_activation
    assert qa(None, 64, p, p, p, n, None) == qk.ERR_INVALID_ARGUMENT
    assert qa(p, 0, p, p, p, n, None) == qk.ERR_INVALID_ARGUMENT
    assert qa(p, 40, p, p, p, n, None) == qk.ERR_UNSUPPORTED
    assert qa(p, 64, ctypes.c_void_p(4097), p, p, n, None) == qk.ERR_MISALIGNED
    assert qa(p, 64, p, p, p, 16, None) == qk.ERR_WORKSPACE_TOO_SMALL
    fq = lib.qkvp_forward_quantized
    dims = qk.Dims(128, 768, 6, 96, 128)
    assert fq(ctypes.byref(dims), 1e-6, p, 128, *([p] * 9), None, 1 << 40, None) == qk.ERR_INVALID_ARGUMENT
    assert fq(ctypes.byref(dims), 1e-6, p, 128, *([p] * 10), 64, None) == qk.ERR_WORKSPACE_TOO_SMALL
    bad = qk.Dims(128, 768, 6, 80, 128)
    assert fq(ctypes.byref(bad), 1e-6, p, 128, *([p] * 10), 1 << 40, None) == qk.ERR_UNSUPPORTED


def test_product_path_refuses_without_library(tmp_path, monkeypatch):
    import fp8_packed_reduced_gb300 as pkg
    monkeypatch.setattr(pkg, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(pkg, "_lib_handle", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        pkg.lib()


def test_package_does_not_import_oracle():
    src = open(os.path.join(ROOT, "fp8_packed_reduced_gb300", "__init__.py")).read()
    assert "oracle" not in re.sub(r'""".*?"""', "", src, flags=re.S)
    for f in os.listdir(os.path.join(ROOT, "fp8_packed_reduced_gb300", "csrc")):
        assert "oracle" not in open(os.path.join(ROOT, "fp8_packed_reduced_gb300", "csrc", f)).read()
