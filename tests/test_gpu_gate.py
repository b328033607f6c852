"""GPU parity of the fused gate (pi_attn_fwd_gated) against the fp64 oracle.

The gate ("pi-Attention" page, section 2.3: a light MLP per token and per head) is read as one
hidden layer of 8 ReLU units on the head's query and a logistic output; the kernel computes it
from the Q tile it has staged and uses it exactly as pi_attn_fwd uses an alpha input.
"""
import numpy as np
import pytest
import torch

import oracle
import structured_sparse_long_gb300 as pa
from structured_sparse_long_gb300 import build as pbuild
from structured_sparse_long_gb300.synth import (MODE_PI, MODE_PI_BIDIR, WORKLOADS, gate_weights,
                                                make_inputs, small_case)

pytestmark = pytest.mark.gpu

BF16 = (2e-2, 5e-3)


@pytest.fixture(scope="module", autouse=True)
def built():
    pbuild.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    pa.load()
    yield
    assert pa.status() == 0


def close(name, gpu, ref, tol):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    max_abs = float(np.abs(g - r).max())
    rel = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300))
    assert max_abs <= tol[0] and rel <= tol[1], f"{name}: max_abs={max_abs:.3e} rel_l2={rel:.3e}"


def run_case(w):
    inp = make_inputs(w, with_dout=False)
    gate = gate_weights(w.H, w.d, seed=w.seed + 100)
    dev = {n: (t.cuda() if t is not None else None) for n, t in inp.items()}
    out, lse, alpha = pa.fwd_gated(dev["q"], dev["k"], dev["v"], tuple(t.cuda() for t in gate), w.k_local,
                                   w.period, w.S, w.mode)
    torch.cuda.synchronize()
    assert pa.status() == 0
    return inp, dev, gate, out, lse, alpha


CASES = [
    # name, B, H, Hkv, N, d, k, period, S, mode
    ("g-pi-d64", 1, 2, 2, 300, 64, 40, 64, 2, MODE_PI),
    ("g-gqa4-d128", 1, 8, 2, 257, 128, 64, 96, 4, MODE_PI),
    ("g-ragged-d128", 2, 2, 2, 333, 128, 100, 150, 3, MODE_PI),
    ("g-bi-d64", 1, 4, 2, 190, 64, 31, 50, 2, MODE_PI_BIDIR),
    ("g-bi-d128", 1, 4, 1, 300, 128, 100, 128, 3, MODE_PI_BIDIR),
]


@pytest.mark.parametrize("spec", CASES, ids=[c[0] for c in CASES])
def test_gated_forward_matches_oracle(spec):
    name, B, H, Hkv, N, d, k, per, S, mode = spec
    w = small_case(name, B, H, Hkv, N, d, k, per, S, mode, "bf16", seed=21)
    inp, _, gate, out, lse, alpha = run_case(w)
    ref_out, ref_lse, ref_alpha = oracle.fwd_gated(inp["q"], inp["k"], inp["v"], gate, k, per, S, mode)
    assert 0.05 < float(np.std(ref_alpha)) and 0.0 < ref_alpha.min() and ref_alpha.max() < 1.0
    close("alpha", alpha.cpu().numpy(), ref_alpha, (1e-5, 1e-5))
    close("out", out.float().cpu().numpy(), ref_out, BF16)
    close("lse", lse.cpu().numpy(), ref_lse, BF16)


def test_gated_forward_equals_forward_with_its_alpha():
    """The gate's alpha, fed to pi_attn_fwd, gives bit-identical out and lse."""
    w = small_case("g-eq", 1, 8, 2, 700, 128, 64, 96, 4, MODE_PI, "bf16", seed=22)
    _, dev, _, out, lse, alpha = run_case(w)
    out2, lse2 = pa.fwd(dev["q"], dev["k"], dev["v"], alpha, w.k_local, w.period, w.S, w.mode)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_gated_c4_matches_oracle():
    """The long-context GQA layer (B1 H16 Hkv4 N65536 d128 k256 pi1024 S4) with the gate fused."""
    w = WORKLOADS["C4"]
    inp, _, gate, out, lse, alpha = run_case(w)
    ref_out, ref_lse, ref_alpha = oracle.fwd_gated(inp["q"], inp["k"], inp["v"], gate, w.k_local,
                                                   w.period, w.S, w.mode)
    close("alpha", alpha.cpu().numpy(), ref_alpha, (1e-5, 1e-5))
    close("out", out.float().cpu().numpy(), ref_out, BF16)
    close("lse", lse.cpu().numpy(), ref_lse, BF16)
