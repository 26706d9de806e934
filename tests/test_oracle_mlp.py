"""Pins for the ReLU-squared MLP oracle (CPU only): library routines (torch
float64 linear and autograd), a brute-force loop, a case whose squared
activations land on E4M3 codes (for the relu(pre) reconstruction), bit-level
bf16 rounding, and shard additivity of the weight gradients."""

import numpy as np
import torch
import torch.nn.functional as F

import oracle


def _bf16_rne_bits(v):
    """Round float32 values to bf16 by integer arithmetic on their bits."""
    b = np.asarray(v, np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    r = ((b + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def _weights(D=128, F_=256, seed=5):
    g = torch.Generator().manual_seed(seed)
    W1 = (torch.randn(F_, D, generator=g) * D ** -0.5).to(torch.bfloat16).float().numpy()
    W2 = (torch.randn(D, F_, generator=g) * F_ ** -0.5).to(torch.bfloat16).float().numpy()
    x = torch.randn(48, D, generator=g).to(torch.bfloat16).float().numpy()
    dout = torch.randn(48, D, generator=g).to(torch.bfloat16).float().numpy()
    return x, W1, W2, dout


def test_bf16_rounding_matches_bit_arithmetic():
    v = np.concatenate([np.random.default_rng(0).standard_normal(10000) * 10.0 ** np.arange(-3, 7).repeat(1000),
                        [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 0.0]])
    np.testing.assert_array_equal(oracle.to_bf16(v), _bf16_rne_bits(v.astype(np.float32)))
    assert oracle.to_bf16([1.0 + 2.0 ** -8])[0] == 1.0            # tie to even
    assert oracle.to_bf16([1.0 + 3 * 2.0 ** -8])[0] == 1.0 + 2.0 ** -6


def test_forward_matches_linear_and_brute_force():
    x, W1, W2, _ = _weights()
    W1_8, _, s1 = oracle.quantize_weight(W1)
    W2_8, _, s2 = oracle.quantize_weight(W2)
    fw = oracle.mlp_forward(x, W1_8, s1, W2_8, s2)
    xh = torch.from_numpy(oracle.dequantize(fw["x8"], fw["x_scale"]))
    w1 = torch.from_numpy(oracle.dequantize(W1_8, s1))
    np.testing.assert_allclose(fw["pre"], F.linear(xh, w1).numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(fw["h"], _bf16_rne_bits(np.maximum(fw["pre"], 0).astype(np.float64) ** 2))
    hh = torch.from_numpy(oracle.dequantize(fw["h8"], fw["h_scale"]))
    w2 = torch.from_numpy(oracle.dequantize(W2_8, s2))
    np.testing.assert_allclose(fw["out"], F.linear(hh, w2).numpy(), rtol=1e-12, atol=1e-12)
    t, d = 3, 17
    acc = sum(float(hh[t, j]) * float(w2[d, j]) for j in range(W2.shape[1]))
    assert abs(acc - fw["out"][t, d]) <= 1e-12 * max(1.0, abs(acc))


def test_relu_reconstruction_and_derivative_exact_case():
    """pre on a grid whose squares land on E4M3 codes at the scale their amax
    gives (amax 4 -> s = fl32(4/448): 4, 1, 0.25 map to codes 448, 112, 28):
    sqrt(h^) is relu(pre) up to the float32 rounding of the scale, and dpre
    equals torch autograd of relu(pre)^2 to the same precision."""
    rng = np.random.default_rng(1)
    pre = rng.choice([-1.0, 0.0, 0.5, 1.0, 2.0], size=(16, 32))
    pre[0, 0] = 2.0
    h = np.maximum(pre, 0) ** 2
    h8, s_h, _ = oracle.quantize(h)
    np.testing.assert_array_equal(oracle.e4m3_decode(h8), h * 112.0)
    np.testing.assert_allclose(np.sqrt(oracle.dequantize(h8, s_h)), np.maximum(pre, 0), rtol=1e-7, atol=0)
    # dh from an exactly representable upstream gradient and weight
    W2 = rng.choice([-1.0, 0.5, 1.0], size=(8, 32))
    W2[0, 0] = 448.0 / 256
    W2_8, _, s2 = oracle.quantize_weight(W2)
    dout = rng.choice([-2.0, 1.0, 0.25], size=(16, 8))
    g8, s_g, _ = oracle.quantize(dout)
    dh = torch.from_numpy(oracle.dequantize(g8, s_g) @ oracle.dequantize(W2_8, s2))
    p = torch.tensor(pre, requires_grad=True)
    (torch.relu(p) ** 2).backward(dh)
    np.testing.assert_allclose(oracle.mlp_dpre(g8, s_g, W2_8, s2, h8, s_h), p.grad.numpy(), rtol=1e-7,
                               atol=1e-12)


def test_grad_gemms_match_autograd_and_shards():
    x, W1, W2, dout = _weights()
    W1_8, _, s1 = oracle.quantize_weight(W1)
    W2_8, _, s2 = oracle.quantize_weight(W2)
    fw = oracle.mlp_forward(x, W1_8, s1, W2_8, s2)
    bw = oracle.mlp_backward(dout, W1_8, s1, W2_8, s2, fw["x8"], fw["x_scale"], fw["h8"], fw["h_scale"])
    xh = torch.tensor(oracle.dequantize(fw["x8"], fw["x_scale"]), requires_grad=True)
    w1 = torch.tensor(oracle.dequantize(W1_8, s1), requires_grad=True)
    hh = torch.tensor(oracle.dequantize(fw["h8"], fw["h_scale"]), requires_grad=True)
    w2 = torch.tensor(oracle.dequantize(W2_8, s2), requires_grad=True)
    dp = torch.from_numpy(oracle.dequantize(bw["dpre8"], bw["dpre_scale"]))
    gg = torch.from_numpy(oracle.dequantize(bw["dout8"], bw["dout_scale"]))
    F.linear(xh, w1).backward(dp)       # the first layer's linear map, fed dpre^
    F.linear(hh, w2).backward(gg)       # the second layer's, fed dout^
    np.testing.assert_allclose(bw["dx"], xh.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(bw["dW1"], w1.grad.numpy(), rtol=1e-12, atol=1e-10)
    np.testing.assert_allclose(bw["dW2"], w2.grad.numpy(), rtol=1e-12, atol=1e-10)
    # dpre is the bf16 rounding of dh * 2 sqrt(h^) with dh fed by dout^ through W_proj^
    np.testing.assert_array_equal(bw["dpre"], _bf16_rne_bits(
        (hh.grad.numpy() * 2.0 * np.sqrt(hh.detach().numpy())).astype(np.float32)))
    parts = [oracle.mlp_grad_gemms(bw["dpre8"][lo:hi], bw["dpre_scale"], bw["dout8"][lo:hi], bw["dout_scale"],
                                   W1_8, s1, fw["x8"][lo:hi], fw["x_scale"], fw["h8"][lo:hi], fw["h_scale"])
             for lo, hi in ((0, 20), (20, 48))]
    np.testing.assert_allclose(parts[0][1] + parts[1][1], bw["dW1"], rtol=1e-12, atol=1e-10)
    np.testing.assert_allclose(parts[0][2] + parts[1][2], bw["dW2"], rtol=1e-12, atol=1e-10)
