"""Pins for the CPU oracle: every function is checked against something other
than itself (closed forms, library routines, brute force, invariants, torch
autograd).  CPU only."""

import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# E4M3 grid
# ----------------------------------------------------------------------------

def test_decode_named_codes():
    named = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x38: 1.0, 0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0,
             0xB8: -1.0, 0xFE: -448.0, 0x81: -(2.0 ** -9)}
    for c, v in named.items():
        assert oracle.e4m3_decode(np.array([c]))[0] == v, hex(c)
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF]))).all()
    z = oracle.e4m3_decode(np.array([0x80]))[0]
    assert z == 0.0 and np.signbit(z)


def test_decode_grid_increasing():
    g = oracle.e4m3_decode(np.arange(127, dtype=np.uint8))
    assert np.all(np.diff(g) > 0)
    assert g[-1] == oracle.E4M3_MAX


def test_decode_matches_torch_view():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_decode(codes.numpy())
    np.testing.assert_array_equal(got, ref)      # treats NaN as equal to NaN
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def _brute_encode(v):
    """Exhaustive nearest search over the 127 non-negative finite values; ties
    to the even code; saturate; sign kept."""
    grid = [oracle.e4m3_decode(np.array([c]))[0] for c in range(127)]
    out = []
    for x in np.asarray(v, np.float64).ravel():
        a = abs(x)
        best, bestd = None, None
        for c, g in enumerate(grid):
            d = abs(a - g)
            if bestd is None or d < bestd or (d == bestd and c % 2 == 0):
                best, bestd = c, d
        out.append(best | (0x80 if np.signbit(x) else 0))
    return np.array(out, dtype=np.uint8)


def test_encode_brute_force():
    rng = np.random.default_rng(0)
    v = np.concatenate([
        rng.standard_normal(400) * 100,
        rng.standard_normal(300) * 2.0 ** -7,
        rng.uniform(-600, 600, 100),
        oracle.e4m3_decode(np.arange(127)),                      # grid points
        (oracle.e4m3_decode(np.arange(126)) + oracle.e4m3_decode(np.arange(1, 127))) / 2,  # midpoints
    ]).astype(np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode(v), _brute_encode(v))


def test_encode_named_ties_and_saturation():
    cases = {2.0 ** -10: 0x00, 3 * 2.0 ** -10: 0x02, 1.0625: 0x38, 1.1875: 0x3A,
             464.0: 0x7E, 470.0: 0x7E, 1e30: 0x7E, -1e30: 0xFE, 448.0: 0x7E,
             -1e-30: 0x80, 0.0: 0x00, 2.0 ** -9: 0x01}
    for v, c in cases.items():
        assert oracle.e4m3_encode(np.array([v], np.float32))[0] == c, v


@pytest.mark.parametrize("scale", [1.0, 0.0078125, 3.7, 1.0 / 448.0, 0.2857142984867096])
def test_encode_matches_torch_cast_all_bf16(scale):
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    v = bits.view(torch.bfloat16).to(torch.float32)
    v = v[torch.isfinite(v)]
    q = (v / torch.tensor(scale, dtype=torch.float32))
    q = q[torch.isfinite(q)]
    ref = q.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(q.numpy())
    np.testing.assert_array_equal(got, ref)


# ----------------------------------------------------------------------------
# Scale and per-tensor quantisation
# ----------------------------------------------------------------------------

def test_scale_closed_form():
    assert oracle.scale_of(448.0) == np.float32(1.0)
    assert oracle.scale_of(0.0) == np.float32(1.0)
    assert oracle.scale_of(1.0) == np.float32(1.0) / np.float32(448.0)
    assert oracle.scale_of(3.5) == np.float32(3.5 / 448.0)


def test_quantize_amax_maps_to_448_and_matches_torch():
    x = synth._normal((64, 256), 1.0, 7)
    codes, s, amax = oracle.quantize(synth.to_numpy_f32(x))
    xf = x.float()
    assert amax == np.float32(xf.abs().max().item())
    ref = (xf / torch.tensor(np.float32(amax) / np.float32(448.0))).clamp(-448, 448)
    ref = ref.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(codes, ref)
    assert (codes & 0x7F).max() == 0x7E          # the amax element hits 448


# ----------------------------------------------------------------------------
# Page-printed shape counts
# ----------------------------------------------------------------------------

def test_page_shape_counts():
    g = json.load(open(os.path.join(GOLDEN, "page_shape_counts.json")))
    assert oracle.packed_width(1, g["d_qk"], g["d_v"]) == g["cols_per_head"]
    assert oracle.packed_width(1, g["d_qk_before"], g["d_v"]) == g["cols_per_head_before"]
    assert round(100 * (1 - g["d_qk"] / g["d_qk_before"]), 1) == g["qk_work_saving_pct"]
    assert round(100 * (1 - g["cols_per_head"] / g["cols_per_head_before"]), 1) == g["qkv_width_saving_pct"]


# ----------------------------------------------------------------------------
# GEMM, norm, RoPE
# ----------------------------------------------------------------------------

def test_packed_gemm_equals_three_projections():
    rng = np.random.default_rng(1)
    H, d_qk, d_v, D, T = 3, 8, 16, 32, 5
    x = rng.standard_normal((T, D))
    Wq, Wk, Wv = (rng.standard_normal((H * d, D)) for d in (d_qk, d_qk, d_v))
    Y = oracle.packed_gemm(x, np.concatenate([Wq, Wk, Wv]))
    (q0, q1), (k0, k1), (v0, v1) = oracle.split_columns(H, d_qk, d_v)
    np.testing.assert_allclose(Y[:, q0:q1], F.linear(torch.tensor(x), torch.tensor(Wq)).numpy(), rtol=1e-13, atol=1e-12)
    np.testing.assert_allclose(Y[:, k0:k1], F.linear(torch.tensor(x), torch.tensor(Wk)).numpy(), rtol=1e-13, atol=1e-12)
    np.testing.assert_allclose(Y[:, v0:v1], F.linear(torch.tensor(x), torch.tensor(Wv)).numpy(), rtol=1e-13, atol=1e-12)


def test_packed_gemm_brute_force():
    rng = np.random.default_rng(2)
    x, W = rng.standard_normal((3, 7)), rng.standard_normal((5, 7))
    Y = oracle.packed_gemm(x, W)
    for t in range(3):
        for n in range(5):
            acc = 0.0
            for d in range(7):
                acc += x[t, d] * W[n, d]
            assert abs(Y[t, n] - acc) < 1e-12


def test_rms_norm_matches_torch_and_unit_rms():
    rng = np.random.default_rng(3)
    Y = rng.standard_normal((2, 9, 96)) * 3.0
    y, r = oracle.rms_norm(Y, 1e-6)
    ref = F.rms_norm(torch.tensor(Y), (96,), eps=1e-6).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    ms = np.mean(Y * Y, axis=-1)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, -1)), np.sqrt(ms / (ms + 1e-6)), rtol=1e-12)
    # scale invariance up to eps
    y2, _ = oracle.rms_norm(7.0 * Y, 1e-6)
    np.testing.assert_allclose(y2, y, rtol=1e-6, atol=1e-7)


def _rope_complex(y, pos, d, base=10000.0):
    """RoPE as multiplication of z = y_i + j y_{i+d/2} by exp(j pos w_i)."""
    half = d // 2
    w = base ** (-(torch.arange(half, dtype=torch.float64) * 2.0) / d)
    ang = torch.tensor(np.asarray(pos, np.float64))[:, None] * w[None, :]
    yt = torch.as_tensor(y)
    z = torch.complex(yt[..., :half], yt[..., half:]) * torch.polar(torch.ones_like(ang), ang)
    return torch.cat([z.real, z.imag], dim=-1).numpy()


@pytest.mark.parametrize("d", [64, 96, 128])
def test_rope_matches_complex_form(d):
    rng = np.random.default_rng(4)
    pos = rng.integers(0, 8192, size=11)
    y = rng.standard_normal((3, 11, d))
    got = oracle.rope(y, oracle.rope_angles(pos, d))
    # angles up to 8191 rad carry ~1e-12 absolute rounding in either formulation
    np.testing.assert_allclose(got, _rope_complex(y, pos, d), rtol=1e-10, atol=1e-10)


def test_rope_invariants():
    rng = np.random.default_rng(5)
    d = 96
    y = rng.standard_normal((4, d))
    pos = np.array([0, 1, 17, 8191])
    th = oracle.rope_angles(pos, d)
    o = oracle.rope(y, th)
    np.testing.assert_allclose(np.linalg.norm(o, axis=-1), np.linalg.norm(y, axis=-1), rtol=1e-12)
    np.testing.assert_allclose(o[0], y[0], rtol=0, atol=0)          # position 0 is the identity
    np.testing.assert_allclose(oracle.rope_inverse(o, th), y, rtol=1e-12, atol=1e-12)
    # a score depends only on the position offset
    a, b = rng.standard_normal(d), rng.standard_normal(d)
    def score(p, pp):
        ta, tb = oracle.rope_angles([p], d), oracle.rope_angles([pp], d)
        return float(oracle.rope(a[None], ta)[0] @ oracle.rope(b[None], tb)[0])
    assert abs(score(3, 10) - score(103, 110)) < 1e-9
    assert abs(score(3, 10) - score(0, 7)) < 1e-9


# ----------------------------------------------------------------------------
# Bank
# ----------------------------------------------------------------------------

def test_quantize_bank_layouts_and_scale():
    [(Wq, Wk, Wv)] = synth.bank_layers(1, H=2, D=128, d_qk=96, d_v=128, seed=11)
    W8, W8T, s = oracle.quantize_bank(*(synth.to_numpy_f32(w) for w in (Wq, Wk, Wv)))
    assert W8.shape == (2 * 320, 128) and W8T.shape == (128, 640)
    np.testing.assert_array_equal(W8T, W8.T)
    W = torch.cat([Wq, Wk, Wv]).float()
    amax = W.abs().max()
    assert s == np.float32(amax.item()) / np.float32(448.0)
    ref = (W / torch.tensor(s)).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(W8, ref)


def test_bank_refresh_changes_with_update():
    [(a, b, c)] = synth.bank_layers(1, H=2, D=128, seed=5)
    [(a2, b2, c2)] = synth.bank_layers(1, H=2, D=128, seed=5, perturb=1e-3)
    W8, _, _ = oracle.quantize_bank(*(synth.to_numpy_f32(w) for w in (a, b, c)))
    W8b, _, _ = oracle.quantize_bank(*(synth.to_numpy_f32(w) for w in (a2, b2, c2)))
    assert (W8 != W8b).any()


# ----------------------------------------------------------------------------
# Forward against a textbook torch layer
# ----------------------------------------------------------------------------

def _torch_layer(x8, s_x, W8, s_w, pos, H, d_qk, d_v, eps=1e-6):
    xh = torch.tensor(x8).view(torch.float8_e4m3fn).double() * float(s_x)
    Wh = torch.tensor(W8).view(torch.float8_e4m3fn).double() * float(s_w)
    Wq, Wk, Wv = Wh.split([H * d_qk, H * d_qk, H * d_v])
    T = xh.shape[0]
    q = F.linear(xh, Wq).view(T, H, d_qk).transpose(0, 1)
    k = F.linear(xh, Wk).view(T, H, d_qk).transpose(0, 1)
    v = F.linear(xh, Wv).view(T, H, d_v).transpose(0, 1)
    q = F.rms_norm(q, (d_qk,), eps=eps)
    k = F.rms_norm(k, (d_qk,), eps=eps)
    return (_rope_complex(q.numpy(), pos, d_qk), _rope_complex(k.numpy(), pos, d_qk), v.numpy())


@pytest.mark.parametrize("d_qk", [128, 96, 64])
def test_forward_matches_textbook_layer(d_qk):
    s = synth.Shape(T=40, D=256, H=2, d_qk=d_qk, d_v=128, seq_len=16)
    inp = synth.forward_inputs(s, seed=3)
    W8, W8T, s_w = oracle.quantize_bank(*(synth.to_numpy_f32(inp[k]) for k in ("Wq", "Wk", "Wv")))
    x = synth.to_numpy_f32(inp["x"])
    pos = inp["pos"].numpy()
    out = oracle.forward(x, W8, s_w, pos, s.H, d_qk, 128)
    q, k, v = _torch_layer(out["x8"], out["x_scale"], W8, s_w, pos, s.H, d_qk, 128)
    np.testing.assert_allclose(out["q"], q, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(out["k"], k, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(out["v"], v, rtol=1e-10, atol=1e-12)
    # x8 equals torch's cast at the same scale
    ref8 = (inp["x"].float() / torch.tensor(out["x_scale"])).clamp(-448, 448)
    np.testing.assert_array_equal(out["x8"], ref8.to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def test_forward_row_subset_matches_full():
    s = synth.Shape(T=64, D=256, H=2, seq_len=32)
    inp = synth.forward_inputs(s, seed=9)
    W8, _, s_w = oracle.quantize_bank(*(synth.to_numpy_f32(inp[k]) for k in ("Wq", "Wk", "Wv")))
    x, pos = synth.to_numpy_f32(inp["x"]), inp["pos"].numpy()
    full = oracle.forward(x, W8, s_w, pos, 2, 96, 128)
    rows = np.array([0, 5, 63, 31])
    sub = oracle.forward(x, W8, s_w, pos, 2, 96, 128, rows=rows)
    for key in ("q", "k", "v"):
        np.testing.assert_array_equal(sub[key], full[key][:, rows])
    np.testing.assert_array_equal(sub["rstd"], full["rstd"][:, :, rows])


# ----------------------------------------------------------------------------
# Backward against torch autograd
# ----------------------------------------------------------------------------

def _autograd_dY(Y, pos, H, d_qk, d_v, dq, dk, dv, eps=1e-6):
    Yt = torch.tensor(Y, requires_grad=True)
    T = Y.shape[0]
    q, k, v = Yt.split([H * d_qk, H * d_qk, H * d_v], dim=1)
    q = F.rms_norm(q.reshape(T, H, d_qk).transpose(0, 1), (d_qk,), eps=eps)
    k = F.rms_norm(k.reshape(T, H, d_qk).transpose(0, 1), (d_qk,), eps=eps)
    v = v.reshape(T, H, d_v).transpose(0, 1)
    half = d_qk // 2
    w = 10000.0 ** (-(torch.arange(half, dtype=torch.float64) * 2.0) / d_qk)
    ang = torch.tensor(np.asarray(pos, np.float64))[:, None] * w
    c, s = torch.cos(ang), torch.sin(ang)
    rot = lambda u: torch.cat([u[..., :half] * c - u[..., half:] * s, u[..., half:] * c + u[..., :half] * s], -1)
    loss = (rot(q) * torch.tensor(dq)).sum() + (rot(k) * torch.tensor(dk)).sum() + (v * torch.tensor(dv)).sum()
    loss.backward()
    return Yt.grad.numpy()


def test_epilogue_backward_matches_autograd():
    s = synth.Shape(T=24, D=256, H=2, d_qk=96, d_v=128, seq_len=24)
    inp = synth.forward_inputs(s, seed=21)
    g = synth.backward_inputs(s, seed=21)
    W8, _, s_w = oracle.quantize_bank(*(synth.to_numpy_f32(inp[k]) for k in ("Wq", "Wk", "Wv")))
    pos = inp["pos"].numpy()
    fw = oracle.forward(synth.to_numpy_f32(inp["x"]), W8, s_w, pos, s.H, 96, 128)
    dq, dk, dv = (synth.to_numpy_f32(g[k]).astype(np.float64) for k in ("dq", "dk", "dv"))
    dY = oracle.epilogue_backward(dq, dk, dv, fw["q"], fw["k"], fw["rstd"], pos, s.H, 96, 128)
    ref = _autograd_dY(fw["Y"], pos, s.H, 96, 128, dq, dk, dv)
    np.testing.assert_allclose(dY, ref, rtol=1e-9, atol=1e-11)


def test_dyq_orthogonality_closed_form():
    rng = np.random.default_rng(8)
    d, T = 96, 6
    Y = rng.standard_normal((1, T, d)) * 0.01      # small rms so eps matters
    y, r = oracle.rms_norm(Y, 1e-6)
    th = oracle.rope_angles(np.arange(T), d)
    out = oracle.rope(y, th)
    dout = rng.standard_normal((1, T, d))
    dY = oracle.norm_rope_backward(dout, out, r, th)
    g = oracle.rope_inverse(dout, th)
    ms = np.mean(Y * Y, -1)
    lhs = np.sum(dY * y, -1)
    rhs = r * np.sum(g * y, -1) * 1e-6 / (ms + 1e-6)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-7, atol=1e-12)


def test_grad_gemms_match_autograd_and_shard():
    rng = np.random.default_rng(10)
    T, D, N = 16, 64, 40
    x8 = oracle.e4m3_encode(rng.standard_normal((T, D)) * 30).astype(np.uint8)
    W8 = oracle.e4m3_encode(rng.standard_normal((N, D)) * 30).astype(np.uint8)
    dY8 = oracle.e4m3_encode(rng.standard_normal((T, N)) * 30).astype(np.uint8)
    s_x, s_w, s_dy = np.float32(0.01), np.float32(0.002), np.float32(0.3)
    dX, dW = oracle.grad_gemms(dY8, s_dy, W8, s_w, x8, s_x)
    xh = torch.tensor(x8).view(torch.float8_e4m3fn).double().mul(float(s_x)).requires_grad_()
    Wh = torch.tensor(W8).view(torch.float8_e4m3fn).double().mul(float(s_w)).requires_grad_()
    dYh = torch.tensor(dY8).view(torch.float8_e4m3fn).double() * float(s_dy)
    F.linear(xh, Wh).backward(dYh)
    np.testing.assert_allclose(dX, xh.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dW, Wh.grad.numpy(), rtol=1e-12, atol=1e-12)
    # dW is additive over token shards
    acc = np.zeros_like(dW)
    for sl in (slice(0, 5), slice(5, 11), slice(11, 16)):
        acc += oracle.grad_gemms(dY8[sl], s_dy, W8, s_w, x8[sl], s_x)[1]
    np.testing.assert_allclose(acc, dW, rtol=1e-12, atol=1e-12)


def test_backward_saved_state_reading():
    """With bf16-rounded saved outputs the backward stays close to the exact one
    (the rebuilt y differs only by the bf16 rounding of the saved q/k)."""
    s = synth.Shape(T=32, D=256, H=2, seq_len=32)
    inp = synth.forward_inputs(s, seed=4)
    g = synth.backward_inputs(s, seed=4)
    W8, _, s_w = oracle.quantize_bank(*(synth.to_numpy_f32(inp[k]) for k in ("Wq", "Wk", "Wv")))
    pos = inp["pos"].numpy()
    fw = oracle.forward(synth.to_numpy_f32(inp["x"]), W8, s_w, pos, 2, 96, 128)
    dq, dk, dv = (synth.to_numpy_f32(g[k]) for k in ("dq", "dk", "dv"))
    exact = oracle.epilogue_backward(dq, dk, dv, fw["q"], fw["k"], fw["rstd"], pos, 2, 96, 128)
    qb = torch.tensor(fw["q"]).to(torch.bfloat16).double().numpy()
    kb = torch.tensor(fw["k"]).to(torch.bfloat16).double().numpy()
    rb = fw["rstd"].astype(np.float32)
    approx = oracle.epilogue_backward(dq, dk, dv, qb, kb, rb, pos, 2, 96, 128)
    rel = np.linalg.norm(approx - exact) / np.linalg.norm(exact)
    assert rel < 2e-3
