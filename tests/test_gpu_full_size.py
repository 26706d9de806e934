"""Parity at the full training shape (6 x 8192 tokens, D = 768, H = 6,
d_qk = 96, d_v = 128) in the launch configuration the benchmark times.

The oracle computes what is cheap at this size in full (scales, the backward
epilogue, its codes, dW) and the rest on sampled token rows."""

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_chain_close, assert_close, assert_codes_match

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
f32 = synth.to_numpy_f32
DEV = "cuda:0"


@pytest.fixture(scope="module")
def run():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_packed_reduced_gb300 import build as b
    b.build()
    import fp8_packed_reduced_gb300 as qk
    s = synth.TRAIN
    inp = synth.forward_inputs(s, seed=0)
    g = synth.backward_inputs(s, seed=0)
    layers = [tuple(inp[k].to(DEV) for k in ("Wq", "Wk", "Wv"))]
    W8, W8T, w_scale = qk.quantize_bank(layers, s.H)
    table = qk.build_rope_table(s.seq_len, s.d_qk, 10000.0, DEV)
    ws = qk.new_workspace(qk.Shape(s.T, s.D, s.H), DEV)
    q, k, v, saved = qk.forward(inp["x"].to(DEV), inp["pos"].to(DEV), W8[0], w_scale[0:1], s.H, table, ws=ws)
    out = qk.backward(*(g[n].to(DEV) for n in ("dq", "dk", "dv")), saved, W8T[0], w_scale[0:1], table, ws=ws)
    torch.cuda.synchronize()
    assert qk.poll_device_status(ws) == (qk.OK, 0)
    res = dict(q=q.cpu(), k=k.cpu(), v=v.cpu(), rstd=saved.rstd.cpu(), x8=saved.x8.cpu(),
               x_scale=saved.x_scale.item(), W8=W8[0].cpu().numpy(), W8T=W8T[0].cpu().numpy(),
               w_scale=w_scale[0].item(), **{n: out[n].cpu() for n in ("dx", "dW", "dY8")},
               dy_scale=out["dy_scale"].item())
    return s, inp, g, res


ROWS = np.unique(np.concatenate([np.arange(0, 64), np.arange(8150, 8250), np.arange(49152 - 64, 49152),
                                 np.random.default_rng(0).integers(0, 49152, 400)]))


def test_bank_and_activation_codes(run):
    s, inp, g, r = run
    oW8, oW8T, os_w = oracle.quantize_bank(*(f32(inp[k]) for k in ("Wq", "Wk", "Wv")))
    np.testing.assert_array_equal(r["W8"], oW8)
    np.testing.assert_array_equal(r["W8T"], oW8T)
    assert r["w_scale"] == float(os_w)
    xf = f32(inp["x"])
    s_x = oracle.scale_of(np.max(np.abs(xf)))
    assert r["x_scale"] == float(s_x)
    x8 = r["x8"].numpy()
    np.testing.assert_array_equal(x8[ROWS], oracle.quantize_with_scale(xf[ROWS], s_x))


def test_forward_sampled_rows(run):
    s, inp, g, r = run
    oW8, _, os_w = oracle.quantize_bank(*(f32(inp[k]) for k in ("Wq", "Wk", "Wv")))
    fw = oracle.forward(f32(inp["x"]), oW8, os_w, inp["pos"].numpy(), s.H, s.d_qk, s.d_v, rows=ROWS)
    for name in ("q", "k", "v"):
        assert_close(f32(r[name][:, ROWS]), fw[name], name)
    assert_close(r["rstd"][:, :, ROWS].numpy(), fw["rstd"], "rstd")


def test_backward_full_codes_and_sampled_gradients(run):
    s, inp, g, r = run
    pos = inp["pos"].numpy()
    # the backward from the GPU's saved state (bf16 q, k; float32 rstd)
    dY = oracle.epilogue_backward(f32(g["dq"]), f32(g["dk"]), f32(g["dv"]), f32(r["q"]), f32(r["k"]),
                                  r["rstd"].numpy(), pos, s.H, s.d_qk, s.d_v)
    dY8_ref, s_dy, _ = oracle.quantize(dY)
    assert abs(r["dy_scale"] - float(s_dy)) <= 1e-6 * float(s_dy)
    dY8 = r["dY8"].numpy()
    assert_codes_match(dY8, dY8_ref, "dY8")
    oW8, _, os_w = oracle.quantize_bank(*(f32(inp[k]) for k in ("Wq", "Wk", "Wv")))
    x8 = r["x8"].numpy()
    # dX on sampled rows and dW in full, from the GPU's codes
    dYh = oracle.dequantize(dY8[ROWS], np.float32(r["dy_scale"]))
    assert_close(f32(r["dx"][ROWS]), dYh @ oracle.dequantize(oW8, os_w), "dx")
    _, dW = oracle.grad_gemms(dY8, np.float32(r["dy_scale"]), oW8, os_w, x8, np.float32(r["x_scale"]))
    assert_close(f32(r["dW"]), dW, "dW")
    # and the whole chain from the oracle's own codes and scale: dX on the
    # sampled rows, dW in full (see assert_chain_close)
    agree = bool(np.array_equal(dY8, dY8_ref))
    dYh_ref = oracle.dequantize(dY8_ref[ROWS], s_dy)
    assert_chain_close(f32(r["dx"][ROWS]), dYh_ref @ oracle.dequantize(oW8, os_w), "dx (oracle's own codes)",
                       bool(np.array_equal(dY8[ROWS], dY8_ref[ROWS])))
    _, dW_ref = oracle.grad_gemms(dY8_ref, s_dy, oW8, os_w, x8, np.float32(r["x_scale"]))
    assert_chain_close(f32(r["dW"]), dW_ref, "dW (oracle's own codes)", agree)


def test_backward_repeatable(run):
    """Three more backward passes on the same inputs give bit-identical codes
    and gradients: the stage ring, the code staging and the split-K reduction
    leave no room for ordering races at this size."""
    import fp8_packed_reduced_gb300 as qk
    s, inp, g, r = run
    dev_in = [g[n].to(DEV) for n in ("dq", "dk", "dv")]
    saved = qk.Saved(q=r["q"].to(DEV), k=r["k"].to(DEV), rstd=r["rstd"].to(DEV), x8=r["x8"].to(DEV),
                     x_scale=torch.tensor([r["x_scale"]], dtype=torch.float32, device=DEV),
                     pos=inp["pos"].to(DEV))
    W8T = torch.from_numpy(r["W8T"]).to(DEV)
    w_scale = torch.tensor([r["w_scale"]], dtype=torch.float32, device=DEV)
    table = qk.build_rope_table(s.seq_len, s.d_qk, 10000.0, DEV)
    for _ in range(3):
        out = qk.backward(*dev_in, saved, W8T, w_scale, table)
        torch.cuda.synchronize()
        assert out["dy_scale"].item() == r["dy_scale"]
        assert torch.equal(out["dY8"].cpu(), r["dY8"])
        assert torch.equal(out["dx"].cpu(), r["dx"])
        assert torch.equal(out["dW"].cpu(), r["dW"])
