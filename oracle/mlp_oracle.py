"""Plain CPU oracle for the FP8 ReLU-squared MLP, forward and backward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the test-suite, ``__graft_entry__.smoke()`` and the
CPU legs of ``bench.py`` use it.  It shares no code with the CUDA library; it
reuses the per-tensor E4M3 quantiser of ``qkvp_oracle`` (pinned there).

What it computes, and where it comes from:

  [PR] "Track 1 (1.167 min on 8xH100, -5.15% same-node): Reduced-width QK and
       packed FP8 attention", section "Changes": FP8 extended to the whole
       ReLU-squared MLP, forward and backward, over all of its GEMMs; the
       saved pre-activation is dropped because relu(pre) can be recovered from
       the stored squared activation (also in the review comments, where the
       author describes the change).
  The MLP: pre = x . W_fc^T, h = relu(pre)^2, out = h . W_proj^T, with
  W_fc [F, D] and W_proj [D, F] stored out x in (F the hidden width).

Readings taken where the pages leave a step open:

  * FP8 recipe of the packed projection: OCP E4M3FN, one per-tensor scale
    amax / 448 (float32) per operand (x, W_fc, h, W_proj, dout, dpre).
  * h reaches FP8 through the activation precision: a per-tensor scale needs
    the amax of all of h before any code, so h is materialised in bf16
    (rounded to nearest even) and quantised from there; the stored squared
    activation of the backward is that FP8 copy (h8 and its scale).
  * relu(pre) is recovered as sqrt(h^) from the de-quantised stored h^, so
    dpre = dh * 2 sqrt(h^), with dh = dout^ . W_proj^; dpre is likewise
    rounded to bf16 and quantised with its own scale.
  * dx = dpre^ . W_fc^, dW_fc = dpre^^T . x^, dW_proj = dout^^T . h^; the
    quantisers are straight-through.
  * Decisions that produce codes are taken in float32 (the kernels'
    precision) on values first rounded to bf16.

All other arithmetic is float64.

Pins (CPU tests, against something other than this file): torch float64
autograd of the same MLP (quantisers as identity) for the chain rule and the
ReLU-squared derivative; relu(p) = sqrt(relu(p)^2) exactly for the bf16 grid
of h; a brute-force loop on a tiny case; dW additivity over token shards.
"""

from __future__ import annotations

import numpy as np
import torch

from .qkvp_oracle import dequantize, quantize


def to_bf16(v) -> np.ndarray:
    """Round to bf16 (nearest even) and return the values as float64."""
    t = torch.from_numpy(np.asarray(v, np.float64).astype(np.float32))
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def mlp_forward(x, W1_8, s_1, W2_8, s_2):
    """x [T, D] (bf16 values); W1_8 [F, D], W2_8 [D, F] codes with scales.

    Returns dict(out [T, D] float64, x8, x_scale, pre [T, F] float64,
    h [T, F] (bf16 values), h8, h_scale)."""
    x8, s_x, _ = quantize(x)
    pre = dequantize(x8, s_x) @ dequantize(W1_8, s_1).T
    h = to_bf16(np.maximum(pre, 0.0) ** 2)
    h8, s_h, _ = quantize(h)
    out = dequantize(h8, s_h) @ dequantize(W2_8, s_2).T
    return dict(out=out, x8=x8, x_scale=s_x, pre=pre, h=h, h8=h8, h_scale=s_h)


def mlp_dpre(dout8, s_g, W2_8, s_2, h8, s_h):
    """dpre = (dout^ . W_proj^) * 2 sqrt(h^) in float64, before rounding."""
    dh = dequantize(dout8, s_g) @ dequantize(W2_8, s_2)
    return dh * 2.0 * np.sqrt(dequantize(h8, s_h))


def mlp_grad_gemms(dpre8, s_p, dout8, s_g, W1_8, s_1, x8, s_x, h8, s_h):
    """dx = dpre^ . W_fc^, dW_fc = dpre^^T . x^, dW_proj = dout^^T . h^."""
    dp = dequantize(dpre8, s_p)
    return (dp @ dequantize(W1_8, s_1), dp.T @ dequantize(x8, s_x),
            dequantize(dout8, s_g).T @ dequantize(h8, s_h))


def mlp_backward(dout, W1_8, s_1, W2_8, s_2, x8, s_x, h8, s_h):
    """Backward from the saved FP8 state (x8, h8 and their scales).

    Returns dict(dx [T, D], dW1 [F, D], dW2 [D, F] float64, dout8, dout_scale,
    dpre (bf16 values), dpre8, dpre_scale)."""
    g8, s_g, _ = quantize(dout)
    dpre = to_bf16(mlp_dpre(g8, s_g, W2_8, s_2, h8, s_h))
    p8, s_p, _ = quantize(dpre)
    dx, dW1, dW2 = mlp_grad_gemms(p8, s_p, g8, s_g, W1_8, s_1, x8, s_x, h8, s_h)
    return dict(dx=dx, dW1=dW1, dW2=dW2, dout8=g8, dout_scale=s_g, dpre=dpre, dpre8=p8, dpre_scale=s_p)
