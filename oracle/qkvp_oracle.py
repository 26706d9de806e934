"""Plain CPU oracle for the reduced-width packed FP8 QKV projection.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the test-suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code, table or constant
generator with the CUDA library and imports nothing from it.

What it computes, and where each step comes from:

  [96] "96 is enough: shrinking attention's routing vectors", section "The change":
       the three projections are packed into one bank (W_packed = concat of
       W_q, W_k, W_v along the output dimension, 96 + 96 + 128 = 320 columns
       per head), one FP8 matmul gives qkv, it is split into [d_qk, d_qk, d_v],
       q and k are RMS-normalised ("direction is all that survives") and then
       rotated by RoPE.
  [PR] "Track 1 (1.167 min on 8xH100, -5.15% same-node): Reduced-width QK and
       packed FP8 attention", section "Changes": Q/K width 96, V 128; packed QKV
       in one FP8 operation; row-major and transposed FP8 weight layouts cached
       once per optimizer update from one weight read; QK norm + RoPE + layout
       conversion fused; the logical Q/K/V packs are quantised without
       materialising a concatenation.  Section "Speed": the backward is FP8 too.
  [8s] "Where the eight seconds were hiding", section "The inventory": tensors
       stay in FP8 across the packed path; both views of the bank are cached.

Readings taken where the pages leave a step open (each is also listed in the
design notes of the repository):

  * FP8 format: OCP E4M3FN (bias 7, largest finite 448, no infinities).  One
    per-tensor scale s = amax / 448 computed in float32; amax == 0 gives s = 1.
  * Encoding: code = E(float32(v) / float32(s)) with float32 IEEE division,
    E = round-to-nearest-even onto the E4M3 grid, saturating to +-448, the sign
    kept (a negative value that rounds to zero encodes as 0x80).
  * Bank order [all-heads Q; all-heads K; all-heads V]; head h is a contiguous
    slice of each block.  W is stored [out, in]; qkv = x . W^T.
  * One scale for x, one per layer for the whole bank, one for dY.
  * RMSNorm has no gain; eps = 1e-6 inside the square root; applied per
    (token, head) to q and to k after de-quantisation; V is not normalised.
  * RoPE is rotate-half over all d_qk/2 frequencies,
    inv_freq_i = base^(-2 i / d_qk) with base 10000; angles in float64; the
    position is the index inside its own sequence.
  * Backward: the exact chain rule of the forward at the point described by
    the saved state (bf16 q/k outputs and float32 rstd): y = RoPE^T(q_out),
    dY_q = r (g - y . mean(g * y)) with g = RoPE^T(dq); dY_v = dv.  dY is
    quantised like the forward operands; dX = dY^ . W^, dW = dY^^T . x^.
    The quantisers are straight-through.
  * Decisions that produce integer codes are taken in float32 (the precision
    the kernels use): values are rounded to float32 before the division.

All real arithmetic other than those float32 decisions is float64.

Pins (each checked by a CPU test against something other than this file):
  e4m3_decode    closed form on named codes; strictly increasing grid;
                 torch's float8_e4m3fn view of all 256 codes.
  e4m3_encode    exhaustive nearest-value search with ties to the even code;
                 torch's float8_e4m3fn cast of every finite bf16 pattern
                 (after clamping to +-448) at several scales; named ties.
  scale_of       closed form amax/448 and the amax == 0 rule.
  packed GEMM    equals three separate projections; brute-force triple loop.
  rms_norm       torch.nn.functional.rms_norm (float64); unit-RMS invariant.
  rope           complex-exponential formulation; norm preservation;
                 identity at position 0; scores depend on position offset only.
  forward        d_qk = 128 equals a textbook torch float64 layer.
  backward       torch float64 autograd of the same forward; <dY_q, y> closed
                 form; dW additivity over token shards.
The pages print no numeric worked example for any of these functions, so no
pin comes from a value printed on the pages.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0  # largest finite E4M3FN value: 1.75 * 2**8


# ----------------------------------------------------------------------------
# E4M3FN grid
# ----------------------------------------------------------------------------

def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3FN byte, as float64 (NaN for 0x7F / 0xFF).

    Layout of a byte: sign bit 7, exponent bits 6..3 (bias 7), mantissa bits
    2..0.  Exponent field 0 is subnormal: m * 2**-9.  Otherwise
    (1 + m/8) * 2**(e-7).  Exponent 15 with mantissa 7 is NaN; there is no
    infinity, so 0x7E = 448 is the largest finite value.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    sub = m.astype(np.float64) * 2.0 ** -9
    nrm = (1.0 + m.astype(np.float64) / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    val = np.where(e == 0, sub, nrm)
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


def _positive_grid():
    """The 127 finite non-negative E4M3FN values (codes 0x00..0x7E), ascending,
    and the 126 midpoints between neighbours (exact in float64)."""
    grid = e4m3_decode(np.arange(0, 127, dtype=np.uint8))
    mids = (grid[:-1] + grid[1:]) / 2.0
    return grid, mids


_GRID, _MIDS = _positive_grid()


def e4m3_encode(values) -> np.ndarray:
    """Round float values onto E4M3FN: nearest grid value, ties to the even
    code, saturating magnitudes above 448 to 448, sign kept.

    Input is taken as given (float32 in practice); NaN/inf are out of contract.
    The magnitude's code is the number of midpoints strictly below it, moved
    up by one when it sits exactly on a midpoint and the upper neighbour has
    the even code.
    """
    v = np.asarray(values, dtype=np.float64)
    a = np.abs(v)
    below = np.searchsorted(_MIDS, a, side="left")          # midpoints < a
    on_mid = np.zeros(a.shape, dtype=bool)
    inside = below < _MIDS.size
    on_mid[inside] = _MIDS[below[inside]] == a[inside]
    # on a midpoint between code k=below and k+1: pick the even one
    code = np.where(on_mid & (below % 2 == 1), below + 1, below)
    code = np.minimum(code, 126).astype(np.uint8)           # saturate to 448
    neg = np.signbit(v)
    return np.where(neg, code | 0x80, code).astype(np.uint8)


# ----------------------------------------------------------------------------
# Per-tensor quantisation
# ----------------------------------------------------------------------------

def scale_of(amax) -> np.float32:
    """Per-tensor scale s = amax / 448 in float32 (s = 1 when amax == 0)."""
    a = np.float32(amax)
    if a == 0:
        return np.float32(1.0)
    return np.float32(a / np.float32(E4M3_MAX))


def quantize(values):
    """Quantise one tensor with its own per-tensor scale.

    Returns (codes uint8 with the shape of ``values``, scale float32, amax
    float32).  Values are first rounded to float32 (the precision in which the
    kernels take the decision), amax is exact over those float32 values, and
    each code is E(v / s) with float32 division.
    """
    v32 = np.asarray(values, dtype=np.float64).astype(np.float32)
    amax = np.float32(np.max(np.abs(v32))) if v32.size else np.float32(0.0)
    s = scale_of(amax)
    return quantize_with_scale(v32, s), s, amax


def quantize_with_scale(values, s) -> np.ndarray:
    """codes = E(float32(v) / float32(s)) elementwise."""
    v32 = np.asarray(values, dtype=np.float64).astype(np.float32)
    q = (v32 / np.float32(s)).astype(np.float32)   # IEEE float32 division
    return e4m3_encode(q)


def dequantize(codes, s) -> np.ndarray:
    """code -> value * s in float64."""
    return e4m3_decode(codes) * np.float64(s)


# ----------------------------------------------------------------------------
# Shapes
# ----------------------------------------------------------------------------

def packed_width(H: int, d_qk: int, d_v: int) -> int:
    """Rows of the packed bank: H heads of (d_qk + d_qk + d_v) columns."""
    return H * (2 * d_qk + d_v)


def split_columns(H: int, d_qk: int, d_v: int):
    """Column ranges of the q, k and v blocks in the packed output."""
    nq = H * d_qk
    return (0, nq), (nq, 2 * nq), (2 * nq, 2 * nq + H * d_v)


# ----------------------------------------------------------------------------
# Bank refresh ("once per optimizer update", both layouts from one read)
# ----------------------------------------------------------------------------

def quantize_bank(Wq, Wk, Wv):
    """Quantise one layer's logical Q/K/V packs as a single bank.

    Wq [H*d_qk, D], Wk [H*d_qk, D], Wv [H*d_v, D] hold bf16 values (passed as
    float32/float64).  The bank is their concatenation along the output
    dimension; one scale covers the whole bank.  Returns
    (W8 [N, D] uint8, W8T [D, N] uint8, s_w float32).
    """
    W = np.concatenate([np.asarray(Wq, np.float64), np.asarray(Wk, np.float64),
                        np.asarray(Wv, np.float64)], axis=0)
    W8, s_w, _ = quantize(W)
    return W8, np.ascontiguousarray(W8.T), s_w


# ----------------------------------------------------------------------------
# RoPE and RMSNorm
# ----------------------------------------------------------------------------

def rope_angles(pos, d_qk: int, base: float = 10000.0) -> np.ndarray:
    """theta[t, i] = pos[t] * base^(-2 i / d_qk), i < d_qk/2, in float64."""
    half = d_qk // 2
    inv_freq = np.power(np.float64(base), -2.0 * np.arange(half, dtype=np.float64) / d_qk)
    return np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]


def rope(y, theta) -> np.ndarray:
    """Rotate-half RoPE along the last axis.

    y [..., T, d]; theta [T, d/2].  For i < d/2:
      o_i       = y_i cos - y_{i+d/2} sin
      o_{i+d/2} = y_{i+d/2} cos + y_i sin
    """
    half = y.shape[-1] // 2
    c, s = np.cos(theta), np.sin(theta)
    a, b = y[..., :half], y[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def rope_inverse(o, theta) -> np.ndarray:
    """The transpose (= inverse) of ``rope``: rotation by -theta."""
    half = o.shape[-1] // 2
    c, s = np.cos(theta), np.sin(theta)
    a, b = o[..., :half], o[..., half:]
    return np.concatenate([a * c + b * s, b * c - a * s], axis=-1)


def rms_norm(Y, eps: float = 1e-6):
    """y = Y * r, r = 1 / sqrt(mean(Y^2) + eps) along the last axis (no gain).
    Returns (y, r) with r of shape Y.shape[:-1]."""
    r = 1.0 / np.sqrt(np.mean(Y * Y, axis=-1) + eps)
    return Y * r[..., None], r


# ----------------------------------------------------------------------------
# Forward
# ----------------------------------------------------------------------------

def packed_gemm(x_hat, W_hat) -> np.ndarray:
    """Y = x^ . W^^T in float64 (the single packed projection)."""
    return np.asarray(x_hat, np.float64) @ np.asarray(W_hat, np.float64).T


def forward(x, W8, s_w, pos, H, d_qk, d_v, eps=1e-6, base=10000.0,
            rows=None, x_scale=None):
    """Packed QKV forward.

    x    [T, D] bf16 values (float32 array); W8 [N, D] codes; s_w float32.
    pos  [T] int positions.
    rows optional token indices: compute only those tokens (the scale of x is
         still taken over all of x unless ``x_scale`` is given).

    Returns a dict:
      q [H, Tr, d_qk], k [H, Tr, d_qk], v [H, Tr, d_v]   float64
      rstd [2, H, Tr]                                     float64 (q then k)
      x8 [Tr, D] codes, x_scale float32, x_amax float32
      y_q, y_k [H, Tr, d_qk]   normalised, pre-RoPE (float64)
      Y [Tr, N]                de-quantised packed GEMM output (float64)
    """
    x = np.asarray(x)
    if x_scale is None:
        amax = np.float32(np.max(np.abs(x.astype(np.float32))))
        s_x = scale_of(amax)
    else:
        s_x, amax = np.float32(x_scale), np.float32(np.nan)
    idx = np.arange(x.shape[0]) if rows is None else np.asarray(rows)
    xr = x[idx]
    x8 = quantize_with_scale(xr, s_x)
    Y = packed_gemm(dequantize(x8, s_x), dequantize(W8, s_w))
    (q0, q1), (k0, k1), (v0, v1) = split_columns(H, d_qk, d_v)
    Tr = len(idx)
    heads = lambda blk, d: blk.reshape(Tr, H, d).transpose(1, 0, 2)
    Yq, Yk, Yv = heads(Y[:, q0:q1], d_qk), heads(Y[:, k0:k1], d_qk), heads(Y[:, v0:v1], d_v)
    yq, rq = rms_norm(Yq, eps)
    yk, rk = rms_norm(Yk, eps)
    theta = rope_angles(np.asarray(pos)[idx], d_qk, base)
    c = np.ascontiguousarray
    return dict(q=c(rope(yq, theta)), k=c(rope(yk, theta)), v=c(Yv),
                rstd=c(np.stack([rq, rk])), x8=x8, x_scale=s_x, x_amax=amax,
                y_q=c(yq), y_k=c(yk), Y=Y)


# ----------------------------------------------------------------------------
# Backward
# ----------------------------------------------------------------------------

def norm_rope_backward(d_out, out_saved, r, theta):
    """Gradient w.r.t. the pre-norm projection Y of out = RoPE(Y * r).

    d_out, out_saved [H, T, d]; r [H, T]; theta [T, d/2].
    y = RoPE^T(out_saved), g = RoPE^T(d_out), dY = r (g - y mean(g*y)).
    """
    y = rope_inverse(np.asarray(out_saved, np.float64), theta)
    g = rope_inverse(np.asarray(d_out, np.float64), theta)
    m = np.mean(g * y, axis=-1, keepdims=True)
    return np.asarray(r, np.float64)[..., None] * (g - y * m)


def epilogue_backward(dq, dk, dv, q_saved, k_saved, rstd, pos, H, d_qk, d_v,
                      base=10000.0):
    """dY [T, N] (float64) in the packed column order from the upstream
    gradients of q, k ([H, T, d_qk]) and v ([H, T, d_v])."""
    theta = rope_angles(pos, d_qk, base)
    rstd = np.asarray(rstd, np.float64)
    dYq = norm_rope_backward(dq, q_saved, rstd[0], theta)
    dYk = norm_rope_backward(dk, k_saved, rstd[1], theta)
    T = theta.shape[0]
    tok = lambda a, d: np.asarray(a, np.float64).transpose(1, 0, 2).reshape(T, H * d)
    return np.concatenate([tok(dYq, d_qk), tok(dYk, d_qk), tok(dv, d_v)], axis=1)


def grad_gemms(dY8, s_dy, W8, s_w, x8, s_x):
    """dX = dY^ . W^ ([T, D]) and dW = dY^^T . x^ ([N, D]) in float64."""
    dYh = dequantize(dY8, s_dy)
    dX = dYh @ dequantize(W8, s_w)
    dW = dYh.T @ dequantize(x8, s_x)
    return dX, dW


def backward(dq, dk, dv, q_saved, k_saved, rstd, pos, W8, s_w, x8, s_x,
             H, d_qk, d_v, base=10000.0):
    """Packed QKV backward: epilogue backward, FP8 quantisation of dY, and the
    two gradient GEMMs.  Returns a dict with dX [T, D], dW [N, D] (float64),
    dY [T, N] (float64, before quantisation), dY8 [T, N] codes, dy_scale."""
    dY = epilogue_backward(dq, dk, dv, q_saved, k_saved, rstd, pos, H, d_qk, d_v, base)
    dY8, s_dy, amax = quantize(dY)
    dX, dW = grad_gemms(dY8, s_dy, W8, s_w, x8, s_x)
    return dict(dX=dX, dW=dW, dY=dY, dY8=dY8, dy_scale=s_dy, dy_amax=amax)
