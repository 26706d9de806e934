"""GPU parity of the FP8 output projection over the V/O bank, through the C
ABI, against the CPU oracle on the same seeded inputs.  Codes and scales are
bit-exact; outputs satisfy max|err| <= 2e-2 * rms(ref) and relative Frobenius
error <= 5e-3."""

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_close

pytestmark = pytest.mark.gpu
f32 = synth.to_numpy_f32
DEV = "cuda:0"


@pytest.fixture(scope="module")
def qk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_packed_reduced_gb300 import build as b
    b.build()
    import fp8_packed_reduced_gb300 as pkg
    pkg.lib()
    return pkg


# (T, D, K): the workload's widths (K = H * d_v = D at H = 6), a ragged token
# tail, one token, output widths that are not multiples of 256, wide K
SHAPES = [(128, 768, 768), (200, 768, 768), (1, 768, 768), (300, 640, 768), (260, 1024, 640),
          (384, 2048, 1024)]
IDS = [f"T{t}_D{d}_K{k}" for t, d, k in SHAPES]


def _run(qk, T, D, K, seed=0):
    inp = synth.oproj_inputs(T, D, K, seed)
    Wo = inp["Wo"].to(DEV)
    W8, W8T, s_o = qk.quantize_weight([Wo])
    ws = qk.new_oproj_workspace(T, D, K, DEV)
    out, a8, a_scale = qk.oproj_forward(inp["a"].to(DEV), W8[0], s_o[0:1], ws=ws)
    g = qk.oproj_backward(inp["dout"].to(DEV), W8T[0], s_o[0:1], a8, a_scale, ws=ws)
    torch.cuda.synchronize()
    assert qk.poll_device_status(ws) == (qk.OK, 0)
    return inp, dict(W8=W8[0].cpu().numpy(), W8T=W8T[0].cpu().numpy(), s_o=s_o[0].item(), out=f32(out),
                     a8=a8.cpu().numpy(), a_scale=a_scale.item(), da=f32(g["da"]), dWo=f32(g["dWo"]),
                     dout8=g["dout8"].cpu().numpy(), dout_scale=g["dout_scale"].item())


def _check(qk, T, D, K):
    inp, r = _run(qk, T, D, K)
    oW8, oW8T, os_o = oracle.quantize_weight(f32(inp["Wo"]))
    np.testing.assert_array_equal(r["W8"], oW8)
    np.testing.assert_array_equal(r["W8T"], oW8T)
    assert r["s_o"] == float(os_o)
    fw = oracle.oproj_forward(f32(inp["a"]), oW8, os_o)
    np.testing.assert_array_equal(r["a8"], fw["a8"])
    assert r["a_scale"] == float(fw["a_scale"])
    assert_close(r["out"], fw["out"], "out")
    bw = oracle.oproj_backward(f32(inp["dout"]), oW8, os_o, fw["a8"], fw["a_scale"])
    np.testing.assert_array_equal(r["dout8"], bw["dout8"])
    assert r["dout_scale"] == float(bw["dout_scale"])
    assert_close(r["da"], bw["da"], "da")
    assert_close(r["dWo"], bw["dWo"], "dWo", bf16_rounding=T == 1)


@pytest.mark.parametrize("T,D,K", SHAPES, ids=IDS)
def test_oproj_matches_oracle(qk, T, D, K):
    _check(qk, T, D, K)


@pytest.mark.parametrize("mask", [0, 7])
def test_oproj_cta_pair_masks(qk, mask):
    prev = qk.set_cta_pairs(mask)
    try:
        _check(qk, 200, 768, 768)
        _check(qk, 130, 640, 768)
    finally:
        qk.set_cta_pairs(prev)


def test_oproj_deterministic(qk):
    _, a = _run(qk, 1000, 768, 768, seed=4)
    _, b = _run(qk, 1000, 768, 768, seed=4)
    for name in ("out", "da", "dWo", "a8", "dout8"):
        np.testing.assert_array_equal(a[name], b[name], err_msg=name)


@pytest.mark.slow
def test_oproj_full_size_sampled(qk):
    """The workload's size (6 x 8192 tokens, D = K = 768), in the benchmark's
    launch configuration: scales and codes in full, out and da on sampled
    token rows, dWo in full."""
    T, D, K = 49152, 768, 768
    inp, r = _run(qk, T, D, K)
    oW8, _, os_o = oracle.quantize_weight(f32(inp["Wo"]))
    a, dout = f32(inp["a"]), f32(inp["dout"])
    a8, s_a, _ = oracle.quantize(a)
    g8, s_g, _ = oracle.quantize(dout)
    assert r["a_scale"] == float(s_a) and r["dout_scale"] == float(s_g)
    np.testing.assert_array_equal(r["a8"], a8)
    np.testing.assert_array_equal(r["dout8"], g8)
    rows = np.unique(np.concatenate([np.arange(64), np.arange(T - 64, T),
                                     np.random.default_rng(1).integers(0, T, 400)]))
    out_ref = oracle.dequantize(a8[rows], s_a) @ oracle.dequantize(oW8, os_o).T
    assert_close(r["out"][rows], out_ref, "out (sampled rows)")
    da_ref, _ = oracle.oproj_grad_gemms(g8[rows], s_g, oW8, os_o, a8[rows], s_a)
    assert_close(r["da"][rows], da_ref, "da (sampled rows)")
    _, dWo_ref = oracle.oproj_grad_gemms(g8, s_g, oW8, os_o, a8, s_a)
    assert_close(r["dWo"], dWo_ref, "dWo")


@pytest.mark.parametrize("R,C", [(768, 768), (3072, 768), (640, 1024)])
def test_weight_refresh_several_matrices(qk, R, C):
    """Three matrices in one call: each with its own scale, codes bit-exact in
    both layouts, and the transposed layout a byte-for-byte transpose."""
    g = torch.Generator().manual_seed(R + C)
    mats = [((torch.randn(R, C, generator=g) * (0.5 + i)) * C ** -0.5).to(torch.bfloat16) for i in range(3)]
    W8, W8T, s = qk.quantize_weight([m.to(DEV) for m in mats])
    torch.cuda.synchronize()
    for i, m in enumerate(mats):
        o8, o8T, os_ = oracle.quantize_weight(f32(m))
        np.testing.assert_array_equal(W8[i].cpu().numpy(), o8)
        np.testing.assert_array_equal(W8T[i].cpu().numpy(), o8T)
        assert s[i].item() == float(os_)
