"""GPU parity of pi_attn_decode: one new query per (batch entry, head) against a KV cache.

The decode step is row N-1 of the forward ("pi-Attention: Periodic Sparse Transformers for
Efficient Long-Context Modeling", section 2.1-2.3, causal form; ECP page, section 2), so the
oracle reference is oracle.fwd on a query tensor whose row N-1 holds the new queries, asked
for that row only.  Cases cover one to many 32-key chunks, ragged last chunks, skip rows far
back in the cache, GQA groups of 1 to 16 heads, ECP, both head sizes, and batch sizes that
give clusters of 1 to 8 CTAs.
"""
import numpy as np
import pytest
import torch

import oracle
import structured_sparse_long_gb300 as pa
from structured_sparse_long_gb300 import build as pbuild
from structured_sparse_long_gb300.synth import MODE_ECP, MODE_PI

pytestmark = pytest.mark.gpu

TOL_ABS, TOL_REL = 2e-2, 5e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    pbuild.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    pa.load()
    yield
    assert pa.status() == 0


def draw(B, H, Hkv, N, d, mode, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, N, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, N, d, generator=g).to(torch.bfloat16)
    a = None if mode == MODE_ECP else torch.sigmoid(torch.randn(B, H, generator=g)).float()
    return q, k, v, a


def reference(q, k, v, a, kl, per, S, mode):
    B, H, d = q.shape
    N = k.shape[2]
    qf = torch.zeros(B, H, N, d, dtype=torch.bfloat16)
    qf[:, :, N - 1] = q
    af = None
    if a is not None:
        af = torch.full((B, H, N), 0.5, dtype=torch.float32)
        af[:, :, N - 1] = a
    out, lse = oracle.fwd(qf, k, v, af, kl, per, S, mode, rows=(N - 1, N))
    return out[:, :, 0], lse[:, :, 0]


def close(name, got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{name}: -inf pattern differs"
    diff = np.abs(got[fin] - ref[fin])
    max_abs = float(diff.max()) if diff.size else 0.0
    den = float(np.linalg.norm(ref[fin]))
    rel = float(np.linalg.norm(got[fin] - ref[fin]) / den) if den > 0 else 0.0
    assert max_abs <= TOL_ABS and rel <= TOL_REL, f"{name}: max_abs={max_abs:.3e} rel={rel:.3e}"


CASES = [
    # name, B, H, Hkv, N, d, k_local, period, S, mode
    ("one-key", 2, 4, 2, 1, 64, 8, 4, 2, MODE_PI),
    ("short", 3, 4, 4, 20, 64, 40, 16, 2, MODE_PI),
    ("ragged-chunks", 2, 8, 2, 1000, 128, 100, 150, 3, MODE_PI),
    ("gqa4-c4-like", 2, 16, 4, 5000, 128, 256, 1024, 4, MODE_PI),
    ("gqa16", 1, 16, 1, 3000, 64, 64, 512, 5, MODE_PI),
    ("mha", 4, 8, 8, 700, 64, 31, 50, 4, MODE_PI),
    ("overlap", 2, 2, 2, 400, 64, 40, 16, 5, MODE_PI),
    ("k0", 2, 4, 2, 300, 128, 0, 7, 5, MODE_PI),
    ("S0", 2, 4, 2, 300, 64, 70, 1, 0, MODE_PI),
    ("far-skips", 1, 4, 2, 20000, 64, 32, 4000, 4, MODE_PI),
    ("big-batch", 64, 4, 2, 300, 64, 64, 96, 2, MODE_PI),
    ("ecp", 2, 4, 2, 777, 64, 128, 0, 0, MODE_ECP),
    ("ecp-d128-seg-start", 2, 4, 4, 513, 128, 256, 0, 0, MODE_ECP),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_decode_matches_oracle(case):
    name, B, H, Hkv, N, d, kl, per, S, mode = case
    q, k, v, a = draw(B, H, Hkv, N, d, mode, seed=N + B)
    dev = [t.cuda() if t is not None else None for t in (q, k, v, a)]
    out, lse = pa.decode(*dev, kl, per, S, mode)
    torch.cuda.synchronize()
    assert pa.status() == 0
    ro, rl = reference(q, k, v, a, kl, per, S, mode)
    close("out", out.float().cpu().numpy(), ro)
    close("lse", lse.cpu().numpy(), rl)


def test_decode_equals_last_forward_row():
    """The decode step and the full forward agree on row N-1 (two kernels, one definition)."""
    B, H, Hkv, N, d, kl, per, S = 2, 8, 2, 2048, 128, 256, 512, 3
    q, k, v, a = draw(B, H, Hkv, N, d, MODE_PI, seed=3)
    g = torch.Generator().manual_seed(4)
    qf = torch.randn(B, H, N, d, generator=g).to(torch.bfloat16)
    qf[:, :, N - 1] = q
    af = torch.sigmoid(torch.randn(B, H, N, generator=g)).float()
    af[:, :, N - 1] = a
    out_f, lse_f = pa.fwd(qf.cuda(), k.cuda(), v.cuda(), af.cuda(), kl, per, S, MODE_PI)
    out_d, lse_d = pa.decode(q.cuda(), k.cuda(), v.cuda(), a.cuda(), kl, per, S, MODE_PI)
    torch.cuda.synchronize()
    assert pa.status() == 0
    close("out", out_d.float().cpu().numpy(), out_f[:, :, N - 1].float().cpu().numpy())
    close("lse", lse_d.cpu().numpy(), lse_f[:, :, N - 1].cpu().numpy())


def test_decode_alpha_edges():
    """alpha = 0 with no skip row: no finite logit -> out 0, lse -inf; alpha = 1: skips off."""
    B, H, Hkv, N, d, kl, per, S = 1, 4, 2, 100, 64, 10, 200, 2   # period > N: no skip row
    q, k, v, a = draw(B, H, Hkv, N, d, MODE_PI, seed=8)
    a[0, 0] = 0.0
    a[0, 1] = 1.0
    dev = [t.cuda() for t in (q, k, v, a)]
    out, lse = pa.decode(*dev, kl, per, S, MODE_PI)
    torch.cuda.synchronize()
    assert pa.status() == 0
    assert torch.all(out[0, 0] == 0) and lse[0, 0].item() == float("-inf")
    ro, rl = reference(q, k, v, a, kl, per, S, MODE_PI)
    close("out", out.float().cpu().numpy(), ro)
    close("lse", lse.cpu().numpy(), rl)


def test_decode_at_the_d4_shape():
    """The benchmarked decode step itself: D4's seeded inputs (64 sequences, 16 heads on 4 KV
    heads, cache 16384, d 128, k 256, pi 1024, S 4) in the launch configuration the bench times.
    Row N-1 attends only to the cache rows from N-1 - S*pi on, and the neighbour sets are the same
    in any window that holds them, so the oracle runs on the last S*pi + 1 rows of the cache."""
    from structured_sparse_long_gb300.synth import WORKLOADS, make_inputs
    w = WORKLOADS["D4"]
    inp = make_inputs(w, with_dout=False)
    q, k, v, a = inp["q"], inp["k"], inp["v"], inp["alpha"]
    assert tuple(k.shape) == (64, 4, 16384, 128) and tuple(q.shape) == (64, 16, 128)
    out, lse = pa.decode(q.cuda(), k.cuda(), v.cuda(), a.cuda(), w.k_local, w.period, w.S, w.mode)
    torch.cuda.synchronize()
    assert pa.status() == 0
    s0 = w.N - 1 - w.S * w.period
    ro, rl = reference(q, k[:, :, s0:].contiguous(), v[:, :, s0:].contiguous(), a, w.k_local, w.period,
                       w.S, w.mode)
    close("out", out.float().cpu().numpy(), ro)
    close("lse", lse.cpu().numpy(), rl)
