"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs.  Integer work (FP8 codes, layouts, scales) must be
bit-exact; floating-point outputs must satisfy max|err| <= 2e-2 * rms(ref)
and relative Frobenius error <= 5e-3."""

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_chain_close, assert_close, assert_codes_match

pytestmark = pytest.mark.gpu

f32 = synth.to_numpy_f32


@pytest.fixture(scope="module")
def qk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fp8_packed_reduced_gb300 import build as b
    b.build()
    import fp8_packed_reduced_gb300 as pkg
    pkg.lib()
    return pkg


DEV = "cuda:0"


def _bank(qk, inp, s):
    layers = [tuple(inp[k].to(DEV) for k in ("Wq", "Wk", "Wv"))]
    W8, W8T, w_scale = qk.quantize_bank(layers, s.H, s.d_qk, s.d_v)
    oW8, oW8T, os_w = oracle.quantize_bank(*(f32(inp[k]) for k in ("Wq", "Wk", "Wv")))
    return (W8[0], W8T[0], w_scale[0:1]), (oW8, oW8T, os_w)


def _run_forward(qk, s, seed=0):
    inp = synth.forward_inputs(s, seed=seed)
    (W8, W8T, w_scale), (oW8, oW8T, os_w) = _bank(qk, inp, s)
    table = qk.build_rope_table(s.seq_len, s.d_qk, 10000.0, DEV)
    x, pos = inp["x"].to(DEV), inp["pos"].to(DEV)
    ws = qk.new_workspace(qk.Shape(s.T, s.D, s.H, s.d_qk, s.d_v), DEV)
    q, k, v, saved = qk.forward(x, pos, W8, w_scale, s.H, table, s.d_qk, s.d_v, ws=ws)
    torch.cuda.synchronize()
    return dict(inp=inp, W8=W8, W8T=W8T, w_scale=w_scale, oW8=oW8, os_w=os_w, table=table, ws=ws,
                q=q, k=k, v=v, saved=saved, x8=saved.x8)


SHAPES = [
    synth.TINY,                                                   # T=128, D=768, H=6, 96/96/128
    synth.Shape(T=200, D=768, H=6, d_qk=96, d_v=128, seq_len=64),  # ragged token tail
    synth.Shape(T=1, D=768, H=6, d_qk=96, d_v=128, seq_len=8),     # a single token
    synth.Shape(T=300, D=1024, H=8, d_qk=64, d_v=128, seq_len=256),
    synth.Shape(T=260, D=1024, H=8, d_qk=128, d_v=128, seq_len=256),
    synth.Shape(T=384, D=2048, H=16, d_qk=96, d_v=128, seq_len=384),
    synth.Shape(T=130, D=640, H=5, d_qk=96, d_v=128, seq_len=130),  # odd head count, D % 256 != 0
]
IDS = [f"T{s.T}_D{s.D}_H{s.H}_dqk{s.d_qk}" for s in SHAPES]


# ----------------------------------------------------------------------------
# Bank refresh
# ----------------------------------------------------------------------------

def test_bank_twelve_layers_bit_exact_and_refresh(qk):
    H, D = 6, 768
    layers = synth.bank_layers(12, H=H, D=D, seed=100)
    dev_layers = [tuple(w.to(DEV) for w in l) for l in layers]
    bank = qk.QKVPBank(dev_layers, H)
    torch.cuda.synchronize()
    for l in (0, 5, 11):
        oW8, oW8T, os_w = oracle.quantize_bank(*(f32(w) for w in layers[l]))
        np.testing.assert_array_equal(bank.W8[l].cpu().numpy(), oW8)
        np.testing.assert_array_equal(bank.W8T[l].cpu().numpy(), oW8T)
        assert bank.w_scale[l].item() == float(os_w)
    np.testing.assert_array_equal(bank.W8T.cpu().numpy(), bank.W8.transpose(1, 2).cpu().numpy())
    assert not bank.refresh()                       # nothing changed: cache kept
    # optimizer update: nudge every tensor in place, the cache is refreshed
    upd = synth.bank_layers(12, H=H, D=D, seed=100, perturb=1e-3)
    for l in range(12):
        for j in range(3):
            dev_layers[l][j].copy_(upd[l][j].to(DEV))
    assert bank.refresh() and bank.refreshes == 2
    torch.cuda.synchronize()
    for l in (0, 11):
        oW8, oW8T, os_w = oracle.quantize_bank(*(f32(w) for w in upd[l]))
        np.testing.assert_array_equal(bank.W8[l].cpu().numpy(), oW8)
        np.testing.assert_array_equal(bank.W8T[l].cpu().numpy(), oW8T)
        assert bank.w_scale[l].item() == float(os_w)


@pytest.mark.parametrize("H,D,dqk", [(5, 640, 96), (8, 1024, 64), (3, 384, 128)])
def test_bank_other_shapes(qk, H, D, dqk):
    layers = synth.bank_layers(2, H=H, D=D, d_qk=dqk, seed=7)
    W8, W8T, s = qk.quantize_bank([tuple(w.to(DEV) for w in l) for l in layers], H, dqk, 128)
    for l in range(2):
        oW8, oW8T, os_w = oracle.quantize_bank(*(f32(w) for w in layers[l]))
        np.testing.assert_array_equal(W8[l].cpu().numpy(), oW8)
        np.testing.assert_array_equal(W8T[l].cpu().numpy(), oW8T)
        assert s[l].item() == float(os_w)


# ----------------------------------------------------------------------------
# Forward
# ----------------------------------------------------------------------------

def _check_forward(qk, s):
    r = _run_forward(qk, s)
    inp = r["inp"]
    fw = oracle.forward(f32(inp["x"]), r["oW8"], r["os_w"], inp["pos"].numpy(), s.H, s.d_qk, s.d_v)
    assert r["saved"].x_scale.item() == float(fw["x_scale"])
    np.testing.assert_array_equal(r["x8"].cpu().numpy(), fw["x8"])
    for name in ("q", "k", "v"):
        assert_close(f32(r[name]), fw[name], name)
    assert_close(r["saved"].rstd.cpu().numpy(), fw["rstd"], "rstd")


@pytest.mark.parametrize("s", SHAPES, ids=IDS)
def test_forward_matches_oracle(qk, s):
    _check_forward(qk, s)


def test_split_forward_equals_forward(qk):
    """quantize_activation + forward_quantized give forward()'s results bit for
    bit; the codes are the oracle's."""
    s = synth.Shape(T=300, D=768, H=6, seq_len=256)
    r = _run_forward(qk, s)
    inp = r["inp"]
    x8, sx = qk.quantize_activation(inp["x"].to(DEV), r["ws"])
    q, k, v, saved = qk.forward_quantized(x8, sx, inp["pos"].to(DEV), r["W8"], r["w_scale"], s.H, r["table"],
                                          ws=r["ws"])
    torch.cuda.synchronize()
    assert qk.poll_device_status(r["ws"]) == (qk.OK, 0)
    assert torch.equal(x8, r["x8"]) and sx.item() == r["saved"].x_scale.item()
    for name, t in (("q", q), ("k", k), ("v", v), ("rstd", saved.rstd)):
        assert torch.equal(t, r[name] if name != "rstd" else r["saved"].rstd), name
    codes, scale, _ = oracle.quantize(f32(inp["x"]))
    np.testing.assert_array_equal(x8.cpu().numpy(), codes)
    assert sx.item() == float(scale)


@pytest.mark.parametrize("n", [16, 48, 4096 + 16, 3 * 2 ** 20])
def test_quantize_activation_any_size(qk, n):
    g = torch.Generator().manual_seed(n)
    x = (torch.randn(n, generator=g) * 3).to(torch.bfloat16)
    ws = qk.new_workspace(qk.Shape(128, 768, 6), DEV)
    x8, sx = qk.quantize_activation(x.to(DEV), ws)
    torch.cuda.synchronize()
    assert qk.poll_device_status(ws) == (qk.OK, 0)
    codes, scale, _ = oracle.quantize(f32(x))
    np.testing.assert_array_equal(x8.cpu().numpy(), codes)
    assert sx.item() == float(scale)


def test_forward_deterministic(qk):
    s = synth.Shape(T=520, D=768, H=6, seq_len=512)
    a, b = _run_forward(qk, s), _run_forward(qk, s)
    for name in ("q", "k", "v", "x8"):
        assert torch.equal(a[name], b[name]), name


# ----------------------------------------------------------------------------
# Backward
# ----------------------------------------------------------------------------

def _run_backward(qk, s, seed=0):
    """Backward with the saved state taken from the oracle's forward (rounded
    to the saved precisions), so that both sides start from the same point."""
    r = _run_forward(qk, s, seed)
    inp = r["inp"]
    pos = inp["pos"].numpy()
    fw = oracle.forward(f32(inp["x"]), r["oW8"], r["os_w"], pos, s.H, s.d_qk, s.d_v)
    g = synth.backward_inputs(s, seed=seed)
    q_saved = torch.from_numpy(fw["q"]).to(torch.bfloat16).contiguous()
    k_saved = torch.from_numpy(fw["k"]).to(torch.bfloat16).contiguous()
    rstd_saved = torch.from_numpy(fw["rstd"]).to(torch.float32).contiguous()
    saved = qk.Saved(q=q_saved.to(DEV), k=k_saved.to(DEV), rstd=rstd_saved.to(DEV),
                     x8=r["saved"].x8, x_scale=r["saved"].x_scale, pos=inp["pos"].to(DEV))
    out = qk.backward(*(g[n].to(DEV) for n in ("dq", "dk", "dv")), saved, r["W8T"], r["w_scale"], r["table"],
                      ws=r["ws"])
    torch.cuda.synchronize()
    bw = oracle.backward(*(f32(g[n]) for n in ("dq", "dk", "dv")), f32(q_saved), f32(k_saved),
                         rstd_saved.numpy(), pos, r["oW8"], r["os_w"], fw["x8"], fw["x_scale"],
                         s.H, s.d_qk, s.d_v)
    return out, bw, r, fw


def _check_backward(qk, s):
    out, bw, r, fw = _run_backward(qk, s)
    dy_scale = out["dy_scale"].item()
    assert abs(dy_scale - float(bw["dy_scale"])) <= 1e-6 * float(bw["dy_scale"])
    dY8 = out["dY8"].cpu().numpy()
    assert_codes_match(dY8, bw["dY8"], "dY8")
    # The GEMMs judged on the GPU's own codes: identical inputs, unique result.
    dX, dW = oracle.grad_gemms(dY8, np.float32(dy_scale), r["oW8"], r["os_w"], fw["x8"], fw["x_scale"])
    rank_one = s.T == 1      # dW is an outer product: see assert_close
    assert_close(f32(out["dx"]), dX, "dx (GPU codes)")
    assert_close(f32(out["dW"]), dW, "dW (GPU codes)", bf16_rounding=rank_one)
    # The whole chain against the oracle's own codes (see assert_chain_close:
    # codes on either side of an E4M3 tie are both correct results).
    agree = bool(np.array_equal(dY8, bw["dY8"]))
    assert_chain_close(f32(out["dx"]), bw["dX"], "dx (oracle's own codes)", agree)
    assert_chain_close(f32(out["dW"]), bw["dW"], "dW (oracle's own codes)", agree, bf16_rounding=rank_one)


@pytest.mark.parametrize("s", SHAPES, ids=IDS)
def test_backward_matches_oracle(qk, s):
    _check_backward(qk, s)


# The remaining points of the width / scale sweep (d_qk in {64, 96, 128},
# D in {768, 1024, 2048}, H = D / 128) that the shapes above do not cover,
# each with a ragged token tail: forward and backward against the oracle.
SWEEP_SHAPES = [
    synth.Shape(T=260, D=768, H=6, d_qk=64, d_v=128, seq_len=256),
    synth.Shape(T=260, D=768, H=6, d_qk=128, d_v=128, seq_len=256),
    synth.Shape(T=260, D=1024, H=8, d_qk=96, d_v=128, seq_len=256),
    synth.Shape(T=260, D=2048, H=16, d_qk=64, d_v=128, seq_len=256),
    synth.Shape(T=260, D=2048, H=16, d_qk=128, d_v=128, seq_len=256),
]


@pytest.mark.parametrize("s", SWEEP_SHAPES, ids=[f"T{s.T}_D{s.D}_H{s.H}_dqk{s.d_qk}" for s in SWEEP_SHAPES])
def test_sweep_points_match_oracle(qk, s):
    _check_forward(qk, s)
    _check_backward(qk, s)


# The GEMMs on one CTA per tile (the default runs them on 2-CTA clusters):
# every mask must give the oracle's results.
PAIR_SHAPES = [SHAPES[0], SHAPES[1], SHAPES[2], SHAPES[3], SHAPES[6]]


@pytest.mark.parametrize("mask", [0, 5, 2])
@pytest.mark.parametrize("s", PAIR_SHAPES, ids=[f"T{s.T}_D{s.D}_H{s.H}_dqk{s.d_qk}" for s in PAIR_SHAPES])
def test_cta_pair_masks_match_oracle(qk, s, mask):
    prev = qk.set_cta_pairs(mask)
    try:
        _check_forward(qk, s)
        _check_backward(qk, s)
    finally:
        qk.set_cta_pairs(prev)


def test_gradient_gemms_on_the_same_codes(qk):
    """dX and dW from the GPU's own dY8 codes: isolates the two GEMMs."""
    s = synth.Shape(T=640, D=768, H=6, seq_len=640)
    out, bw, r, fw = _run_backward(qk, s, seed=3)
    dX, dW = oracle.grad_gemms(out["dY8"].cpu().numpy(), np.float32(out["dy_scale"].item()), r["oW8"], r["os_w"],
                               fw["x8"], fw["x_scale"])
    assert_close(f32(out["dx"]), dX, "dx (same codes)")
    assert_close(f32(out["dW"]), dW, "dW (same codes)")


def test_backward_deterministic(qk):
    s = synth.Shape(T=1000, D=768, H=6, seq_len=1000)
    a, _, _, _ = _run_backward(qk, s, seed=5)
    b, _, _, _ = _run_backward(qk, s, seed=5)
    for name in ("dx", "dW", "dY8"):
        assert torch.equal(a[name], b[name]), name


def _step_outputs(qk, inp, g, W8, W8T, w_scale, table, ws, H):
    q, k, v, saved = qk.forward(inp["x"], inp["pos"], W8, w_scale, H, table, ws=ws)
    out = qk.backward(g["dq"], g["dk"], g["dv"], saved, W8T, w_scale, table, ws=ws)
    return dict(q=q, k=k, v=v, rstd=saved.rstd, x8=saved.x8, dY8=out["dY8"], dx=out["dx"], dW=out["dW"])


def test_captured_step_replays_the_same_results(qk):
    """Forward + backward replayed from a captured CUDA graph (as the bench
    times it) give the bits of the same calls made eagerly."""
    s = synth.Shape(T=1000, D=768, H=6, seq_len=1000)
    inp = {n: t.to(DEV) for n, t in synth.forward_inputs(s, seed=7).items()}
    g = {n: t.to(DEV) for n, t in synth.backward_inputs(s, seed=7).items()}
    W8, W8T, w_scale = qk.quantize_bank([(inp["Wq"], inp["Wk"], inp["Wv"])], s.H)
    table = qk.build_rope_table(8192, s.d_qk, 10000.0, DEV)
    ws = qk.new_workspace(qk.Shape(s.T, s.D, s.H), DEV)
    args = (inp, g, W8[0], W8T[0], w_scale[0:1], table, ws, s.H)
    eager = _step_outputs(qk, *args)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        _step_outputs(qk, *args)   # warm-up outside the capture
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            captured = _step_outputs(qk, *args)
    graph.replay()
    torch.cuda.synchronize()
    assert qk.poll_device_status(ws) == (qk.OK, 0)
    for name, t in eager.items():
        assert torch.equal(t, captured[name]), name


# ----------------------------------------------------------------------------
# Device-side error reporting (no fault, no hang)
# ----------------------------------------------------------------------------

def test_wait_timeout_is_reported_and_context_survives(qk):
    ws = qk.new_workspace(qk.Shape(128, 768, 6), DEV)
    assert qk.poll_device_status(ws) == (qk.OK, 0)
    qk.selftest_wait_timeout(ws, 2000)         # a barrier nothing arrives on, 2 ms limit
    code, where = qk.poll_device_status(ws)
    assert code == qk.ERR_TIMEOUT and where == 11
    assert qk.poll_device_status(ws) == (qk.OK, 0)
    # the context is still usable
    r = _run_forward(qk, synth.TINY)
    assert torch.isfinite(r["q"].float()).all()


def test_position_outside_table_is_reported(qk):
    s = synth.TINY
    inp = synth.forward_inputs(s)
    (W8, W8T, w_scale), _ = _bank(qk, inp, s)
    table = qk.build_rope_table(64, s.d_qk, 10000.0, DEV)      # positions reach 127
    ws = qk.new_workspace(qk.Shape(s.T, s.D, s.H), DEV)
    qk.forward(inp["x"].to(DEV), inp["pos"].to(DEV), W8, w_scale, s.H, table, ws=ws)
    code, where = qk.poll_device_status(ws)
    assert code == qk.ERR_DEVICE_INPUT and where == 5


def test_binding_rejects_strided_tensors(qk):
    s = synth.TINY
    r = _run_forward(qk, s)
    g = synth.backward_inputs(s)
    bad = qk.Saved(q=r["q"].transpose(0, 1).contiguous().transpose(0, 1), k=r["k"], rstd=r["saved"].rstd,
                   x8=r["saved"].x8, x_scale=r["saved"].x_scale, pos=r["saved"].pos)
    with pytest.raises(ValueError, match="contiguous"):
        qk.backward(*(g[n].to(DEV) for n in ("dq", "dk", "dv")), bad, r["W8T"], r["w_scale"], r["table"])
