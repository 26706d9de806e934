"""Pins for the O-projection oracle (CPU only): library routines (torch
float64 F.linear and autograd), brute force on a tiny case, shard additivity,
and agreement with the packed-bank quantiser on a single matrix."""

import numpy as np
import torch
import torch.nn.functional as F

import oracle
import synth


def _case(T=40, D=256, K=128, seed=3):
    g = torch.Generator().manual_seed(seed)
    a = torch.randn(T, K, generator=g).to(torch.bfloat16).float().numpy()
    Wo = (torch.randn(D, K, generator=g) * D ** -0.5).to(torch.bfloat16).float().numpy()
    dout = torch.randn(T, D, generator=g).to(torch.bfloat16).float().numpy()
    return a, Wo, dout


def test_weight_codes_equal_the_bank_quantiser_and_transpose():
    _, Wo, _ = _case()
    W8, W8T, s = oracle.quantize_weight(Wo)
    # a bank whose Q and K packs are empty is the single matrix
    B8, B8T, sb = oracle.quantize_bank(np.zeros((0, Wo.shape[1])), np.zeros((0, Wo.shape[1])), Wo)
    np.testing.assert_array_equal(W8, B8)
    np.testing.assert_array_equal(W8T, W8.T)
    assert s == sb == np.float32(np.float32(np.abs(Wo).max()) / np.float32(448.0))


def test_forward_matches_linear_and_brute_force():
    a, Wo, _ = _case()
    W8, _, s_o = oracle.quantize_weight(Wo)
    fw = oracle.oproj_forward(a, W8, s_o)
    a_hat = torch.from_numpy(oracle.dequantize(fw["a8"], fw["a_scale"]))
    w_hat = torch.from_numpy(oracle.dequantize(W8, s_o))
    ref = F.linear(a_hat, w_hat).numpy()
    np.testing.assert_allclose(fw["out"], ref, rtol=1e-12, atol=1e-12)
    # brute force on a corner of the output
    for t in (0, 7, 39):
        for d in (0, 100, 255):
            acc = 0.0
            for k in range(a.shape[1]):
                acc += float(a_hat[t, k]) * float(w_hat[d, k])
            assert abs(acc - fw["out"][t, d]) <= 1e-12 * max(1.0, abs(acc))
    # the activation codes are the generic per-tensor quantiser's
    a8, s_a, _ = oracle.quantize(a)
    np.testing.assert_array_equal(fw["a8"], a8)
    assert fw["a_scale"] == s_a


def test_backward_matches_autograd_and_shards():
    a, Wo, dout = _case()
    W8, W8T, s_o = oracle.quantize_weight(Wo)
    fw = oracle.oproj_forward(a, W8, s_o)
    bw = oracle.oproj_backward(dout, W8, s_o, fw["a8"], fw["a_scale"])
    # autograd of out = a^ W^T with the upstream gradient g^ (straight-through quantisers)
    a_hat = torch.tensor(oracle.dequantize(fw["a8"], fw["a_scale"]), requires_grad=True)
    w_hat = torch.tensor(oracle.dequantize(W8, s_o), requires_grad=True)
    g_hat = torch.from_numpy(oracle.dequantize(bw["dout8"], bw["dout_scale"]))
    F.linear(a_hat, w_hat).backward(g_hat)
    np.testing.assert_allclose(bw["da"], a_hat.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(bw["dWo"], w_hat.grad.numpy(), rtol=1e-12, atol=1e-10)
    # dW_o over token shards adds up to the whole
    parts = [oracle.oproj_grad_gemms(bw["dout8"][lo:hi], bw["dout_scale"], W8, s_o, fw["a8"][lo:hi],
                                     fw["a_scale"])[1] for lo, hi in ((0, 13), (13, 40))]
    np.testing.assert_allclose(parts[0] + parts[1], bw["dWo"], rtol=1e-12, atol=1e-10)
    # the transposed layout serves the same product
    gh = oracle.dequantize(bw["dout8"], bw["dout_scale"])
    np.testing.assert_allclose(gh @ oracle.dequantize(W8T, s_o).T, bw["da"], rtol=1e-12, atol=1e-12)


def test_workload_shapes_from_the_synthetic_module():
    s = synth.TRAIN
    assert s.H * s.d_v == 768 == s.D      # V/O heads keep 128 columns: the O weight is square here
