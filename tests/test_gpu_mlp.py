"""GPU parity of the FP8 ReLU-squared MLP, through the C ABI, against the CPU
oracle on the same seeded inputs.

Each stage is judged on the GPU's own inputs to that stage, where the result
is unique: codes and scales of a quantisation are bit-exact given the values
quantised; GEMM outputs (and the bf16 intermediates h and dpre) satisfy
max|err| <= 2e-2 * rms(ref) and relative Frobenius error <= 5e-3.  The bf16
intermediates h and dpre are products of heavy-tailed factors (a square, and
dh * 2 sqrt(h)); where the GPU's float32 value and the oracle's float64 value
round to neighbouring bf16 numbers, one rounding step of a large element
alone exceeds 2e-2 * rms, so for those two the max bound also admits one bf16
step per element (the Frobenius bound is unchanged).  The whole
chain is also compared with the oracle's own run (codes within one E4M3 step
and >= 99.9 % identical, outputs within tolerance)."""

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_chain_close, assert_close, assert_codes_match

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


# (T, D, F): the workload's widths (F = 4 D), a ragged token tail, one token,
# D not a multiple of 256, a narrower hidden width
SHAPES = [(128, 768, 3072), (200, 768, 3072), (1, 768, 3072), (300, 640, 2560), (256, 1024, 1536)]
IDS = [f"T{t}_D{d}_F{f}" for t, d, f in SHAPES]


def _run(qk, T, D, F_, seed=0):
    inp = synth.mlp_inputs(T, D, F_, seed)
    W1_8, W1_8T, s1 = qk.quantize_weight([inp["W1"].to(DEV)])
    W2_8, W2_8T, s2 = qk.quantize_weight([inp["W2"].to(DEV)])
    ws = qk.new_mlp_workspace(T, D, F_, DEV)
    fw = qk.mlp_forward(inp["x"].to(DEV), W1_8[0], s1[0:1], W2_8[0], s2[0:1], ws=ws)
    bw = qk.mlp_backward(inp["dout"].to(DEV), W1_8T[0], s1[0:1], W2_8T[0], s2[0:1], fw, ws=ws)
    torch.cuda.synchronize()
    assert qk.poll_device_status(ws) == (qk.OK, 0)
    host = lambda t: f32(t) if t.dtype == torch.bfloat16 else t.cpu().numpy()
    r = {k: host(v) for k, v in list(fw.items()) + list(bw.items())}
    r.update(W1_8=W1_8[0].cpu().numpy(), W1_8T=W1_8T[0].cpu().numpy(), s1=s1[0].item(),
             W2_8=W2_8[0].cpu().numpy(), W2_8T=W2_8T[0].cpu().numpy(), s2=s2[0].item())
    for k in ("x_scale", "h_scale", "dout_scale", "dpre_scale"):
        r[k] = np.float32(r[k][0])
    return inp, r


def _check(qk, T, D, F_):
    inp, r = _run(qk, T, D, F_)
    x, dout = f32(inp["x"]), f32(inp["dout"])
    # weights: codes, layouts and scales
    oW1, oW1T, os1 = oracle.quantize_weight(f32(inp["W1"]))
    oW2, oW2T, os2 = oracle.quantize_weight(f32(inp["W2"]))
    for got, ref in ((r["W1_8"], oW1), (r["W1_8T"], oW1T), (r["W2_8"], oW2), (r["W2_8T"], oW2T)):
        np.testing.assert_array_equal(got, ref)
    assert r["s1"] == float(os1) and r["s2"] == float(os2)
    # forward, stage by stage on the GPU's own inputs
    x8, s_x, _ = oracle.quantize(x)
    np.testing.assert_array_equal(r["x8"], x8)
    assert r["x_scale"] == s_x
    pre = oracle.dequantize(x8, s_x) @ oracle.dequantize(oW1, os1).T
    assert_close(r["h"], oracle.to_bf16(np.maximum(pre, 0) ** 2), "h", bf16_rounding=True)
    h8, s_h, _ = oracle.quantize(r["h"])          # the GPU's h quantised: unique codes
    np.testing.assert_array_equal(r["h8"], h8)
    assert r["h_scale"] == s_h
    assert_close(r["out"], oracle.dequantize(h8, s_h) @ oracle.dequantize(oW2, os2).T, "out")
    # backward, stage by stage
    g8, s_g, _ = oracle.quantize(dout)
    np.testing.assert_array_equal(r["dout8"], g8)
    assert r["dout_scale"] == s_g
    assert_close(r["dpre"], oracle.to_bf16(oracle.mlp_dpre(g8, s_g, oW2, os2, h8, s_h)), "dpre", bf16_rounding=True)
    p8, s_p, _ = oracle.quantize(r["dpre"])
    np.testing.assert_array_equal(r["dpre8"], p8)
    assert r["dpre_scale"] == s_p
    dx, dW1, dW2 = oracle.mlp_grad_gemms(p8, s_p, g8, s_g, oW1, os1, x8, s_x, h8, s_h)
    one = T == 1      # rank-one weight gradients: see assert_close
    assert_close(r["dx"], dx, "dx")
    assert_close(r["dW1"], dW1, "dW1", bf16_rounding=one)
    assert_close(r["dW2"], dW2, "dW2", bf16_rounding=one)
    # the whole chain against the oracle's own run
    fw = oracle.mlp_forward(x, oW1, os1, oW2, os2)
    assert_codes_match(r["h8"], fw["h8"], "h8 (oracle's own run)")
    assert_close(r["out"], fw["out"], "out (oracle's own run)")
    bw = oracle.mlp_backward(dout, oW1, os1, oW2, os2, fw["x8"], fw["x_scale"], fw["h8"], fw["h_scale"])
    assert_codes_match(r["dpre8"], bw["dpre8"], "dpre8 (oracle's own run)")
    # the whole chain (see assert_chain_close: codes on either side of an E4M3
    # tie are both correct results)
    agree = bool(np.array_equal(r["h8"], fw["h8"]) and np.array_equal(r["dpre8"], bw["dpre8"]))
    assert_chain_close(r["dx"], bw["dx"], "dx (oracle's own run)", agree)
    assert_chain_close(r["dW1"], bw["dW1"], "dW1 (oracle's own run)", agree, bf16_rounding=one)
    assert_chain_close(r["dW2"], bw["dW2"], "dW2 (oracle's own run)", agree, bf16_rounding=one)


@pytest.mark.parametrize("T,D,F_", SHAPES, ids=IDS)
def test_mlp_matches_oracle(qk, T, D, F_):
    _check(qk, T, D, F_)


@pytest.mark.parametrize("mask", [0, 7])
def test_mlp_cta_pair_masks(qk, mask):
    prev = qk.set_cta_pairs(mask)
    try:
        _check(qk, 200, 768, 3072)
        _check(qk, 130, 640, 2560)
    finally:
        qk.set_cta_pairs(prev)


def test_mlp_deterministic(qk):
    _, a = _run(qk, 700, 768, 3072, seed=6)
    _, b = _run(qk, 700, 768, 3072, seed=6)
    for name in ("out", "h", "h8", "dx", "dW1", "dW2", "dpre8"):
        np.testing.assert_array_equal(a[name], b[name], err_msg=name)


@pytest.mark.slow
def test_mlp_full_size_sampled(qk):
    """The workload's size (6 x 8192 tokens, D = 768, F = 3072) in the
    benchmark's launch configuration: every quantisation in full on the GPU's
    own values, the GEMM outputs on sampled rows."""
    T, D, F_ = 49152, 768, 3072
    inp, r = _run(qk, T, D, F_)
    x, dout = f32(inp["x"]), f32(inp["dout"])
    oW1, _, os1 = oracle.quantize_weight(f32(inp["W1"]))
    oW2, _, os2 = oracle.quantize_weight(f32(inp["W2"]))
    x8, s_x, _ = oracle.quantize(x)
    np.testing.assert_array_equal(r["x8"], x8)
    h8, s_h, _ = oracle.quantize(r["h"])
    np.testing.assert_array_equal(r["h8"], h8)
    assert r["h_scale"] == s_h
    g8, s_g, _ = oracle.quantize(dout)
    np.testing.assert_array_equal(r["dout8"], g8)
    p8, s_p, _ = oracle.quantize(r["dpre"])
    np.testing.assert_array_equal(r["dpre8"], p8)
    assert r["dpre_scale"] == s_p
    rows = np.unique(np.concatenate([np.arange(64), np.arange(T - 64, T),
                                     np.random.default_rng(2).integers(0, T, 300)]))
    pre = oracle.dequantize(x8[rows], s_x) @ oracle.dequantize(oW1, os1).T
    assert_close(r["h"][rows], oracle.to_bf16(np.maximum(pre, 0) ** 2), "h (sampled rows)", bf16_rounding=True)
    assert_close(r["out"][rows], oracle.dequantize(h8[rows], s_h) @ oracle.dequantize(oW2, os2).T,
                 "out (sampled rows)")
    assert_close(r["dpre"][rows], oracle.to_bf16(oracle.mlp_dpre(g8[rows], s_g, oW2, os2, h8[rows], s_h)),
                 "dpre (sampled rows)", bf16_rounding=True)
    assert_close(r["dx"][rows], oracle.dequantize(p8[rows], s_p) @ oracle.dequantize(oW1, os1), "dx (sampled rows)")
    # weight gradients: sampled output rows, every token
    fr = np.random.default_rng(3).choice(F_, 96, replace=False)
    dr = np.random.default_rng(4).choice(D, 48, replace=False)
    dW1_rows = oracle.dequantize(p8[:, fr], s_p).T @ oracle.dequantize(x8, s_x)
    assert_close(r["dW1"][fr], dW1_rows, "dW1 (sampled rows)")
    dW2_rows = oracle.dequantize(g8[:, dr], s_g).T @ oracle.dequantize(h8, s_h)
    assert_close(r["dW2"][dr], dW2_rows, "dW2 (sampled rows)")
