"""Plain CPU oracle for the FP8 output projection over the V/O bank.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the test-suite, ``__graft_entry__.smoke()`` and the
CPU legs of ``bench.py`` use it.  It shares no code with the CUDA library; it
reuses the per-tensor E4M3 quantiser of ``qkvp_oracle`` (pinned there).

What it computes, and where it comes from:

  [PR] "Track 1 (1.167 min on 8xH100, -5.15% same-node): Reduced-width QK and
       packed FP8 attention", section "Changes": Q/K are stored apart from
       "the rectangular V/O bank" (V and O keep the 128-wide heads, so the O
       weight is a D x H*d_v matrix), and both FP8 weight layouts (row-major
       and transposed) are cached once per optimizer update from one read.
       The step after attention projects the concatenated heads back to the
       model width: out = a . W_o^T.

Readings taken where the pages leave the step open:

  * The O projection runs in FP8 with the recipe of the packed projection:
    OCP E4M3FN codes, one per-tensor scale amax / 448 (float32) for the
    attention output a, one for the weight, one for the upstream gradient.
  * W_o is stored [out, in] = [D, K] with K = H * d_v; out = a . W_o^T.
  * Backward, straight through the quantisers: with g = dout quantised,
    da = g^ . W_o^ and dW_o = g^^T . a^, all products in float64.

Pins (CPU tests, against something other than this file): the forward equals
torch float64 F.linear on the de-quantised operands and a brute-force loop on
a tiny case; the backward equals torch float64 autograd of that linear map;
dW_o is additive over token shards; the weight codes equal the packed-bank
quantiser applied to the single matrix.
"""

from __future__ import annotations

import numpy as np

from .qkvp_oracle import dequantize, quantize


def quantize_weight(W):
    """One weight matrix [R, C] (bf16 values) to E4M3 with one scale, in both
    layouts from one quantisation: (W8 [R, C], W8T [C, R], s)."""
    W8, s, _ = quantize(np.asarray(W, np.float64))
    return W8, np.ascontiguousarray(W8.T), s


def oproj_forward(a, Wo8, s_o):
    """out = a^ . W_o^^T in float64, a [T, K] quantised with its own scale.

    Returns dict(out [T, D] float64, a8 [T, K] codes, a_scale, a_amax)."""
    a8, s_a, amax = quantize(a)
    out = dequantize(a8, s_a) @ dequantize(Wo8, s_o).T
    return dict(out=out, a8=a8, a_scale=s_a, a_amax=amax)


def oproj_grad_gemms(g8, s_g, Wo8, s_o, a8, s_a):
    """da = g^ . W_o^ ([T, K]) and dW_o = g^^T . a^ ([D, K]) in float64."""
    gh = dequantize(g8, s_g)
    return gh @ dequantize(Wo8, s_o), gh.T @ dequantize(a8, s_a)


def oproj_backward(dout, Wo8, s_o, a8, s_a):
    """Backward of the O projection: dout [T, D] quantised with its own scale,
    then the two gradient GEMMs.  Returns dict(da, dWo, dout8, dout_scale)."""
    g8, s_g, amax = quantize(dout)
    da, dWo = oproj_grad_gemms(g8, s_g, Wo8, s_o, a8, s_a)
    return dict(da=da, dWo=dWo, dout8=g8, dout_scale=s_g, dout_amax=amax)
