"""The allocation-free bank refresh, qkvp_quantize_bank_static.

It exists for callers that cannot allocate device memory and so cannot hand
qkvp_quantize_bank a workspace; its scratch is a fixed array inside the
library.  These tests call it through the C ABI and compare it with the
workspace entry point on two calls in a row (the second call reuses the array
the first one left behind).  This file is collected last on purpose."""

import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def qk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_packed_reduced_gb300 import build as b
    b.build()
    import fp8_packed_reduced_gb300 as pkg
    f = pkg.lib().qkvp_quantize_bank_static
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_void_p)] * 3 + [ctypes.c_void_p] * 4
    return pkg


def _static_refresh(qk, layers, H, d_qk=96, d_v=128):
    L, D = len(layers), layers[0][0].shape[1]
    N = H * (2 * d_qk + d_v)
    W8 = torch.empty((L, N, D), dtype=torch.uint8, device=DEV)
    W8T = torch.empty((L, D, N), dtype=torch.uint8, device=DEV)
    s = torch.empty((L,), dtype=torch.float32, device=DEV)
    arr = lambda i: (ctypes.c_void_p * L)(*[ctypes.c_void_p(layers[l][i].data_ptr()) for l in range(L)])
    rc = qk.lib().qkvp_quantize_bank_static(L, D, H, d_qk, d_v, arr(0), arr(1), arr(2),
                                            ctypes.c_void_p(W8.data_ptr()), ctypes.c_void_p(W8T.data_ptr()),
                                            ctypes.c_void_p(s.data_ptr()),
                                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, W8, W8T, s


def test_static_refresh_matches_workspace_refresh_twice(qk):
    H, D = 6, 768
    first = [tuple(w.to(DEV) for w in l) for l in synth.bank_layers(12, H=H, D=D, seed=300)]
    second = [tuple(w.to(DEV) for w in l) for l in synth.bank_layers(5, H=H, D=D, seed=400, perturb=1e-3)]
    for layers in (first, second):
        rc, W8, W8T, s = _static_refresh(qk, layers, H)
        assert rc == qk.OK
        rW8, rW8T, rs = qk.quantize_bank(layers, H)
        torch.cuda.synchronize()
        # codes and scales are integer-exact results: bit-for-bit equality
        assert torch.equal(W8, rW8)
        assert torch.equal(W8T, rW8T)
        np.testing.assert_array_equal(s.cpu().numpy(), rs.cpu().numpy())


def test_static_refresh_rejects_banks_beyond_its_scratch(qk):
    H, D = 2, 128
    layers = [tuple(w.to(DEV) for w in l) for l in synth.bank_layers(1, H=H, D=D, seed=1)] * 129
    rc, *_ = _static_refresh(qk, layers, H)
    assert rc == qk.ERR_UNSUPPORTED
