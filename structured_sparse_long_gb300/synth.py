"""Seeded synthetic inputs for the pi-Attention / ECP attention hot path.

This module only draws random tensors.  It holds none of the attention
arithmetic, so both the CUDA path and the fp64 oracle can be fed from it.

Workloads (shapes from "pi-Attention: Periodic Sparse Transformers for
Efficient Long-Context Modeling", section 2 "Methodology", and "Efficient
Context Propagating Perceiver Architectures...", section 2, PAR block):

  C1  tiny fp32 pi-Attention fwd  B1 H2  Hkv2  N256   d32  k16  pi32   S1
  C2  LM-layer bf16 fwd           B4 H12 Hkv12 N4096  d64  k128 pi256  S1
  C3  ECP paired-segment bf16 fwd B2 H16 Hkv16 N8192  d64  c512 (no skip)
  C4  long-context GQA bf16 fwd   B1 H16 Hkv4  N65536 d128 k256 pi1024 S4
  C5  training fwd+bwd bf16       B2 H16 Hkv16 N16384 d64  k256 pi512  S2
  C6  bidirectional GQA bf16 fwd  B1 H16 Hkv4  N65536 d128 k256 pi1024 S4 (band i-k..i+k,
                                  skips i -/+ m*pi: the general form of the same page, 2.1-2.2)
  C7  bidirectional training bf16 B2 H16 Hkv16 N16384 d64  k256 pi512  S2, fwd+bwd (C5's
                                  shapes in the bidirectional form)
  C8  gated long-context GQA     C4's layer with the fused gate: alpha from the per-head MLP
                                  sigmoid(w2_h . max(0, W1_h q + b1_h) + b2_h), computed in the
                                  forward launch (gate_weights(H, d, seed + 100))
  D4  decode step, C4 layer       B64 H16 Hkv4 cache N16384 d128 k256 pi1024 S4: one new
                                  query per sequence (q [B,H,d], alpha [B,H]) against the cache

Draw order per workload: q, k, v, alpha, dout, from one CPU torch.Generator
seeded with the workload's seed.  Values are drawn in fp32 and then cast to
the workload dtype (bf16 or fp32).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

MODE_PI = 0
MODE_ECP = 1
MODE_PI_BIDIR = 2


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Hkv: int
    N: int
    d: int
    k_local: int          # band width k (pi mode) or half-segment length c (ECP mode)
    period: int           # skip period pi (pi mode), unused in ECP mode
    S: int                # number of skip multiples, 0 in ECP mode
    mode: int             # MODE_PI, MODE_ECP or MODE_PI_BIDIR
    dtype: str            # "f32" or "bf16"
    seed: int
    qkv_scale: str        # "unit": N(0,1); "inv_sqrt_d": N(0,1)/sqrt(d)
    alpha: str            # "uniform(a,b)", "sigmoid(sigma)" or "none"
    backward: bool = False
    description: str = ""
    decode: bool = False  # one new query per (b, h) against a KV cache of N rows (row N-1)
    gate: bool = False    # alpha from the fused gate (weights: gate_weights(H, d, seed + 100))

    @property
    def tokens(self) -> int:
        return self.B * self.N

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "C1": Workload("C1", 1, 2, 2, 256, 32, 16, 32, 1, MODE_PI, "f32", 0, "unit",
                   "uniform(0.2,0.8)",
                   description="tiny fp32 pi-Attention fwd"),
    "C2": Workload("C2", 4, 12, 12, 4096, 64, 128, 256, 1, MODE_PI, "bf16", 1, "inv_sqrt_d",
                   "sigmoid(1.0)",
                   description="LM-layer bf16 pi-Attention fwd (125M-class layer, 12x64 heads)"),
    "C3": Workload("C3", 2, 16, 16, 8192, 64, 512, 0, 0, MODE_ECP, "bf16", 2, "unit", "none",
                   description="ECP paired-segment bf16 fwd, half-segment 512"),
    "C4": Workload("C4", 1, 16, 4, 65536, 128, 256, 1024, 4, MODE_PI, "bf16", 3, "unit",
                   "sigmoid(1.5)",
                   description="long-context GQA bf16 pi-Attention fwd"),
    "C5": Workload("C5", 2, 16, 16, 16384, 64, 256, 512, 2, MODE_PI, "bf16", 4, "unit",
                   "sigmoid(1.0)", backward=True,
                   description="training fwd+bwd bf16 pi-Attention"),
    "C6": Workload("C6", 1, 16, 4, 65536, 128, 256, 1024, 4, MODE_PI_BIDIR, "bf16", 5, "unit",
                   "sigmoid(1.5)",
                   description="long-context GQA bf16 bidirectional pi-Attention fwd"),
    "C7": Workload("C7", 2, 16, 16, 16384, 64, 256, 512, 2, MODE_PI_BIDIR, "bf16", 7, "unit",
                   "sigmoid(1.0)", backward=True,
                   description="training fwd+bwd bf16 bidirectional pi-Attention"),
    "C8": Workload("C8", 1, 16, 4, 65536, 128, 256, 1024, 4, MODE_PI, "bf16", 8, "unit", "none",
                   gate=True, description="long-context GQA bf16 pi-Attention fwd with the fused gate"),
    "D4": Workload("D4", 64, 16, 4, 16384, 128, 256, 1024, 4, MODE_PI, "bf16", 6, "unit",
                   "sigmoid(1.5)", decode=True,
                   description="decode step of the long-context GQA layer, 64 sequences"),
}


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _draw_alpha(gen: torch.Generator, shape, spec: str) -> Optional[torch.Tensor]:
    if spec == "none":
        return None
    if spec.startswith("uniform("):
        lo, hi = (float(x) for x in spec[len("uniform("):-1].split(","))
        return lo + (hi - lo) * torch.rand(shape, generator=gen, dtype=torch.float32)
    if spec.startswith("sigmoid("):
        sigma = float(spec[len("sigmoid("):-1])
        return torch.sigmoid(sigma * torch.randn(shape, generator=gen, dtype=torch.float32))
    if spec.startswith("const("):
        val = float(spec[len("const("):-1])
        return torch.full(shape, val, dtype=torch.float32)
    raise ValueError(f"unknown alpha distribution {spec!r}")


def make_inputs(w: Workload, with_dout: Optional[bool] = None, device="cpu") -> dict:
    """Draw q, k, v, alpha (and dout) for workload ``w``.

    Returns a dict of contiguous tensors: q [B,H,N,d], k and v [B,Hkv,N,d]
    (dtype of the workload), alpha [B,H,N] fp32 or None, dout [B,H,N,d] or None.
    A decode workload has q [B,H,d] and alpha [B,H] instead (k and v are the cache).
    """
    if with_dout is None:
        with_dout = w.backward
    gen = torch.Generator(device="cpu")
    gen.manual_seed(w.seed)
    scale = 1.0 / math.sqrt(w.d) if w.qkv_scale == "inv_sqrt_d" else 1.0
    dt = torch_dtype(w.dtype)

    def normal(shape):
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
        if scale != 1.0:
            x = x * scale
        return x.to(dt)

    if w.decode:  # the new queries and their gates; k, v are the cache
        q = normal((w.B, w.H, w.d))
        k = normal((w.B, w.Hkv, w.N, w.d))
        v = normal((w.B, w.Hkv, w.N, w.d))
        alpha = _draw_alpha(gen, (w.B, w.H), w.alpha)
        dout = None
    else:
        q = normal((w.B, w.H, w.N, w.d))
        k = normal((w.B, w.Hkv, w.N, w.d))
        v = normal((w.B, w.Hkv, w.N, w.d))
        alpha = _draw_alpha(gen, (w.B, w.H, w.N), w.alpha)
        dout = normal((w.B, w.H, w.N, w.d)) if with_dout else None
    out = {"q": q, "k": k, "v": v, "alpha": alpha, "dout": dout}
    if device != "cpu":
        out = {n: (t.to(device) if t is not None else None) for n, t in out.items()}
    return out


def small_case(name="case", B=1, H=2, Hkv=2, N=300, d=64, k_local=40, period=64, S=2,
               mode=MODE_PI, dtype="bf16", seed=11, qkv_scale="unit",
               alpha="sigmoid(1.0)", backward=False) -> Workload:
    """A parity-test workload of arbitrary (small) shape."""
    return Workload(name, B, H, Hkv, N, d, k_local, period, S, mode, dtype, seed, qkv_scale,
                    alpha, backward)


GATE_HIDDEN = 8  # hidden units per head of the fused gate


def gate_weights(H: int, d: int, seed: int):
    """Synthetic weights of the fused gate's per-head MLP: W1 [H, 8, d] ~ N(0, 1/d) drawn in fp32
    and cast to bf16 (the tensor-core operand) and b1 [H, 8] ~ N(0, 1/4), so that for
    unit-variance queries the hidden pre-activations have about unit spread; w2 [H, 8] ~ N(0, 2/8)
    and b2 [H] ~ N(0, 1), fp32, so that the output logit spreads over about one unit and alpha
    covers (0, 1) without saturating."""
    gen = torch.Generator().manual_seed(seed)
    w1 = (torch.randn(H, GATE_HIDDEN, d, generator=gen, dtype=torch.float32) / math.sqrt(d)).to(torch.bfloat16)
    b1 = 0.5 * torch.randn(H, GATE_HIDDEN, generator=gen, dtype=torch.float32)
    w2 = torch.randn(H, GATE_HIDDEN, generator=gen, dtype=torch.float32) * math.sqrt(2.0 / GATE_HIDDEN)
    b2 = torch.randn(H, generator=gen, dtype=torch.float32)
    return w1, b1, w2, b2
