"""Seeded synthetic inputs for the packed QKV projection.

This module only draws random numbers and lays out shapes; it holds none of
the method's arithmetic.  The CPU oracle and the CUDA path both receive their
inputs from here (the oracle as NumPy arrays of the bf16 values, the CUDA path
as torch tensors copied to the device).

Workload recipe (the pages train a GPT-style model; no dataset is needed to
exercise this layer, so every tensor is drawn from the distribution the layer
sees at initialisation):
  x          bf16 N(0, 1)        [T, D]
  W_q, W_k   bf16 N(0, 1/D)      [H*d_qk, D]   (std D^-1/2)
  W_v        bf16 N(0, 1/D)      [H*d_v, D]
  dq, dk     bf16 N(0, 1)        [H, T, d_qk]
  dv         bf16 N(0, 1)        [H, T, d_v]
  pos        int32 t mod seq_len (positions restart at every sequence)
One torch CPU generator per tensor, seeded seed+0, seed+1, ... in the order
x, W_q, W_k, W_v, dq, dk, dv.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Shape:
    T: int
    D: int
    H: int
    d_qk: int = 96
    d_v: int = 128
    seq_len: int = 8192

    @property
    def N(self) -> int:
        return self.H * (2 * self.d_qk + self.d_v)


TINY = Shape(T=128, D=768, H=6, d_qk=96, d_v=128, seq_len=128)
TRAIN = Shape(T=49152, D=768, H=6, d_qk=96, d_v=128, seq_len=8192)


def _normal(shape, std, seed, device="cpu"):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    t = torch.randn(shape, generator=g, dtype=torch.float32, device=device)
    if std != 1.0:
        t = t * std
    return t.to(torch.bfloat16)


def positions(T: int, seq_len: int, device="cpu") -> torch.Tensor:
    return (torch.arange(T, dtype=torch.int64, device=device) % seq_len).to(torch.int32)


def forward_inputs(shape: Shape, seed: int = 0, device="cpu"):
    """x, W_q, W_k, W_v (bf16) and pos (int32)."""
    s = shape
    wstd = s.D ** -0.5
    x = _normal((s.T, s.D), 1.0, seed + 0, device)
    Wq = _normal((s.H * s.d_qk, s.D), wstd, seed + 1, device)
    Wk = _normal((s.H * s.d_qk, s.D), wstd, seed + 2, device)
    Wv = _normal((s.H * s.d_v, s.D), wstd, seed + 3, device)
    return dict(x=x, Wq=Wq, Wk=Wk, Wv=Wv, pos=positions(s.T, s.seq_len, device))


def backward_inputs(shape: Shape, seed: int = 0, device="cpu"):
    """Upstream gradients dq, dk [H, T, d_qk] and dv [H, T, d_v] (bf16)."""
    s = shape
    dq = _normal((s.H, s.T, s.d_qk), 1.0, seed + 4, device)
    dk = _normal((s.H, s.T, s.d_qk), 1.0, seed + 5, device)
    dv = _normal((s.H, s.T, s.d_v), 1.0, seed + 6, device)
    return dict(dq=dq, dk=dk, dv=dv)


def bank_layers(L: int, H: int, D: int, d_qk: int = 96, d_v: int = 128, seed: int = 100,
                perturb: float = 0.0, device="cpu"):
    """L layers of (W_q, W_k, W_v), bf16 N(0, 1/D).  With ``perturb`` > 0 each
    tensor gets a uniform U(-perturb, perturb) nudge (an optimizer update) and
    is rounded back to bf16."""
    out = []
    std = D ** -0.5
    for l in range(L):
        ws = []
        for j, rows in enumerate((H * d_qk, H * d_qk, H * d_v)):
            w = _normal((rows, D), std, seed + 3 * l + j, device)
            if perturb:
                g = torch.Generator(device=device)
                g.manual_seed(seed + 100000 + 3 * l + j)
                u = (torch.rand((rows, D), generator=g, device=device) * 2 - 1) * perturb
                w = (w.float() + u).to(torch.bfloat16)
            ws.append(w)
        out.append(tuple(ws))
    return out


def oproj_inputs(T: int, D: int, K: int, seed: int = 0, device="cpu"):
    """Output projection: the heads' attention outputs a [T, K] ~ N(0, 1),
    W_o [D, K] ~ N(0, 1/K) (fan-in K) and the upstream gradient dout [T, D]
    ~ N(0, 1), all bf16; generators seeded seed+20, +21, +22."""
    return dict(a=_normal((T, K), 1.0, seed + 20, device),
                Wo=_normal((D, K), K ** -0.5, seed + 21, device),
                dout=_normal((T, D), 1.0, seed + 22, device))


def mlp_inputs(T: int, D: int, F: int, seed: int = 0, device="cpu"):
    """ReLU-squared MLP: x [T, D] ~ N(0, 1), W_fc [F, D] ~ N(0, 1/D), W_proj
    [D, F] ~ N(0, 1/F) (fan-in scaling) and dout [T, D] ~ N(0, 1), all bf16;
    generators seeded seed+30 ... seed+33."""
    return dict(x=_normal((T, D), 1.0, seed + 30, device),
                W1=_normal((F, D), D ** -0.5, seed + 31, device),
                W2=_normal((D, F), F ** -0.5, seed + 32, device),
                dout=_normal((T, D), 1.0, seed + 33, device))


def to_numpy_f32(t: torch.Tensor):
    """bf16/float tensor -> float32 NumPy array holding the same values."""
    return t.detach().to("cpu", torch.float32).numpy()
