"""Pins for the oracle's bidirectional pi-Attention (mode 2).

The general, non-causal form of "pi-Attention: Periodic Sparse Transformers for Efficient
Long-Context Modeling", section 2.1 (band i-k .. i+k) and 2.2 (skip keys i - m*pi and
i + m*pi), fused as in 2.3: one softmax over the union, +ln(alpha) on band logits and
+ln(1-alpha) on skip logits.  Keys outside [0, N) do not exist; a skip key inside the band
is a band key (each key once).  The oracle is tied here to a dense brute force, to torch's
scaled_dot_product_attention (symmetric window; full attention), to a closed form at q = 0,
to closed-form counts, to the reversal symmetry of the mask, and to autograd and finite
differences for the backward.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from tests.brute import dense_forward

BIDIR = 2


def rand_case(B, H, Hkv, N, d, seed, alpha_lo=0.05, alpha_hi=0.95):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, N, d, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float64)
    a = (alpha_lo + (alpha_hi - alpha_lo) * torch.rand(B, H, N, generator=g)).float()
    return q, k, v, a


CASES = [
    # (B, H, Hkv, N, d, k_local, period, S)
    (1, 2, 2, 37, 8, 5, 7, 3),
    (2, 4, 2, 41, 6, 3, 9, 2),      # GQA
    (1, 4, 1, 33, 5, 0, 4, 5),      # k = 0
    (1, 2, 2, 30, 4, 10, 4, 4),     # skips overlapping the band are dropped
    (1, 2, 2, 30, 4, 8, 4, 3),      # m*pi == k: band key only
    (1, 3, 3, 25, 7, 30, 6, 2),     # band wider than N
    (1, 2, 2, 19, 3, 4, 100, 2),    # no skip key inside [0, N)
    (1, 2, 2, 23, 4, 2, 5, 0),      # S = 0
]


@pytest.mark.parametrize("case", CASES)
def test_bidir_matches_dense_brute_force(case):
    B, H, Hkv, N, d, kl, per, S = case
    q, k, v, a = rand_case(B, H, Hkv, N, d, seed=N + 3 * d)
    out, lse, P = oracle.fwd(q, k, v, a, kl, per, S, BIDIR, want_P=True)
    bo, bl, bP = dense_forward(q, k, v, a, kl, per, S, BIDIR)
    np.testing.assert_allclose(out, bo.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, bl.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(P, bP.numpy(), atol=1e-12, rtol=0)


def _sdpa(q, k, v, mask=None):
    G = q.shape[1] // k.shape[1]
    return F.scaled_dot_product_attention(q, k.repeat_interleave(G, 1), v.repeat_interleave(G, 1),
                                          attn_mask=mask)


@pytest.mark.parametrize("kl", [0, 3, 16])
def test_bidir_s0_is_symmetric_window_and_alpha_free(kl):
    N = 40
    q, k, v, a = rand_case(1, 4, 2, N, 8, seed=100 + kl)
    i = torch.arange(N).view(N, 1)
    j = torch.arange(N).view(1, N)
    ref = _sdpa(q, k, v, mask=(i - j).abs() <= kl)
    out_a, _ = oracle.fwd(q, k, v, a, kl, 5, 0, BIDIR)
    out_1, _ = oracle.fwd(q, k, v, torch.ones_like(a), kl, 5, 0, BIDIR)
    np.testing.assert_allclose(out_a, ref.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(out_1, ref.numpy(), atol=1e-12, rtol=0)


def test_bidir_wide_band_is_full_attention():
    N = 45
    q, k, v, a = rand_case(2, 2, 2, N, 8, seed=4)
    ref = _sdpa(q, k, v)
    for kl in (N - 1, N + 10):
        out, _ = oracle.fwd(q, k, v, a, kl, 7, 0, BIDIR)
        np.testing.assert_allclose(out, ref.numpy(), atol=1e-12, rtol=0)


def test_bidir_q_zero_closed_form():
    """q = 0: weights alpha on the band, 1 - alpha on the skips (both directions)."""
    B, H, N, d, kl, per, S = 1, 2, 60, 5, 6, 11, 4
    _, k, v, a = rand_case(B, H, H, N, d, seed=19)
    q = torch.zeros(B, H, N, d, dtype=torch.float64)
    out, lse = oracle.fwd(q, k, v, a, kl, per, S, BIDIR)
    for h in range(H):
        for i in range(N):
            lo, hi = max(0, i - kl), min(N - 1, i + kl)
            loc = v[0, h, lo:hi + 1].sum(0)
            sk = [i + s * m * per for m in range(1, S + 1) for s in (-1, 1)
                  if m * per > kl and 0 <= i + s * m * per < N]
            skv = v[0, h, sk].sum(0) if sk else torch.zeros(d, dtype=torch.float64)
            al = float(a[0, h, i])
            den = al * (hi - lo + 1) + (1 - al) * len(sk)
            np.testing.assert_allclose(out[0, h, i], ((al * loc + (1 - al) * skv) / den).numpy(),
                                       atol=1e-13, rtol=0)
            assert abs(lse[0, h, i] - math.log(den)) < 1e-13


def test_bidir_is_symmetric_under_sequence_reversal():
    """The bidirectional neighbour set of i maps onto that of N-1-i under j -> N-1-j, so
    reversing q, k, v and alpha along the sequence reverses out and lse."""
    B, H, Hkv, N, d, kl, per, S = 1, 4, 2, 53, 6, 4, 9, 3
    q, k, v, a = rand_case(B, H, Hkv, N, d, seed=8)
    out, lse = oracle.fwd(q, k, v, a, kl, per, S, BIDIR)
    rq, rk, rv, ra = (t.flip(2) for t in (q, k, v, a))
    out_r, lse_r = oracle.fwd(rq, rk, rv, ra, kl, per, S, BIDIR)
    np.testing.assert_allclose(out_r[:, :, ::-1], out, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse_r[:, :, ::-1], lse, atol=1e-12, rtol=0)


def closed_form_counts(N, kl, per, S):
    cnt = np.zeros(N, dtype=np.int64)
    isum = np.zeros(N, dtype=np.int64)
    for i in range(N):
        lo, hi = max(0, i - kl), min(N - 1, i + kl)
        cnt[i] = hi - lo + 1
        isum[i] = (lo + hi) * (hi - lo + 1) // 2
        for m in range(1, S + 1):
            if m * per <= kl:
                continue
            for j in (i - m * per, i + m * per):
                if 0 <= j < N:
                    cnt[i] += 1
                    isum[i] += j
    return cnt, isum


def closed_form_total(N, kl, per, S):
    """Band pairs: each unordered pair |i-j| = t <= k, t > 0, counts twice, plus the diagonal;
    skip pairs: each offset m*pi > k inside [0, N) counts twice."""
    kk = min(kl, N - 1)
    band = N + 2 * sum(N - t for t in range(1, kk + 1))
    skip = sum(2 * max(0, N - m * per) for m in range(1, S + 1) if m * per > kl)
    return band + skip


@pytest.mark.parametrize("case", [(100, 10, 4, 5), (77, 5, 3, 0), (90, 12, 6, 4), (50, 60, 10, 3),
                                  (65536, 256, 1024, 4), (4096, 128, 256, 1)])
def test_bidir_counts_closed_forms(case):
    N, kl, per, S = case
    cnt, isum = oracle.counts(N, kl, per, S, BIDIR)
    if N <= 5000:
        c2, s2 = closed_form_counts(N, kl, per, S)
        np.testing.assert_array_equal(cnt, c2)
        np.testing.assert_array_equal(isum, s2)
    assert int(cnt.sum()) == closed_form_total(N, kl, per, S)


@pytest.mark.parametrize("case", [(1, 4, 2, 29, 5, 4, 6, 3), (1, 2, 1, 26, 6, 10, 4, 4),
                                  (1, 2, 2, 24, 4, 2, 5, 0)])
def test_bidir_bwd_matches_autograd_through_brute_force(case):
    B, H, Hkv, N, d, kl, per, S = case
    q, k, v, a = rand_case(B, H, Hkv, N, d, seed=2 * N, alpha_lo=0.1, alpha_hi=0.9)
    g = torch.Generator().manual_seed(6)
    dout = torch.randn(B, H, N, d, generator=g, dtype=torch.float64)
    dq, dk, dv, dal = oracle.bwd(q, k, v, a, dout, kl, per, S, BIDIR)
    qt, kt, vt = (t.clone().requires_grad_(True) for t in (q, k, v))
    at = a.double().clone().requires_grad_(True)
    out, _, _ = dense_forward(qt, kt, vt, at, kl, per, S, BIDIR)
    out.backward(dout)
    np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-10, rtol=0)
    np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-10, rtol=0)
    np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-10, rtol=0)
    np.testing.assert_allclose(dal, at.grad.numpy(), atol=1e-9, rtol=1e-9)


def test_bidir_bwd_finite_differences():
    B, H, Hkv, N, d, kl, per, S = 1, 2, 1, 15, 3, 2, 4, 3
    q, k, v, a = rand_case(B, H, Hkv, N, d, seed=41, alpha_lo=0.2, alpha_hi=0.8)
    g = torch.Generator().manual_seed(7)
    dout = torch.randn(B, H, N, d, generator=g, dtype=torch.float64)
    dq, dk, dv, _ = oracle.bwd(q, k, v, a, dout, kl, per, S, BIDIR)
    eps = 1e-6
    rng = np.random.default_rng(1)

    def loss(qq, kk, vv):
        out, _ = oracle.fwd(qq, kk, vv, a, kl, per, S, BIDIR)
        return float((out * dout.numpy()).sum())

    for name, t, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, s)) for s in t.shape)
            tp, tm = t.clone(), t.clone()
            tp[idx] += eps
            tm[idx] -= eps
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = tp, tm
            num = (loss(**{"qq": args_p["q"], "kk": args_p["k"], "vv": args_p["v"]})
                   - loss(**{"qq": args_m["q"], "kk": args_m["k"], "vv": args_m["v"]})) / (2 * eps)
            assert abs(num - grad[idx]) <= 1e-6 * max(1.0, abs(num)), (name, idx, num, grad[idx])
