"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each test ties the oracle to something the pages or the mathematics fix:
brute force over a dense broadcast mask, reductions to torch's
scaled_dot_product_attention, closed forms, invariants, a hand-worked
example and finite differences.  Sources: "pi-Attention: Periodic Sparse
Transformers for Efficient Long-Context Modeling" section 2.1-2.3 (band,
causal pi-skip, one softmax over the union with alpha as log-prior); the ECP
page, section 2 (paired half-segment PAR block); the GSS-Transformer hybrid
page, attention branch (GQA).
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from tests.brute import dense_forward, union_masks

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_case(B, H, Hkv, N, d, seed, alpha_lo=0.05, alpha_hi=0.95, dtype=torch.float64):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, N, d, generator=g, dtype=torch.float64).to(dtype)
    k = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float64).to(dtype)
    v = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float64).to(dtype)
    a = (alpha_lo + (alpha_hi - alpha_lo) * torch.rand(B, H, N, generator=g)).float()
    return q, k, v, a


PI_CASES = [
    # (B, H, Hkv, N, d, k_local, period, S)
    (1, 2, 2, 37, 8, 5, 7, 3),
    (2, 4, 2, 41, 6, 3, 9, 2),      # GQA G=2
    (1, 4, 1, 33, 5, 0, 4, 5),      # k=0: band is the diagonal only
    (1, 2, 2, 30, 4, 10, 4, 4),     # skip overlaps the band: m=1,2 dropped
    (1, 2, 2, 30, 4, 8, 4, 3),      # m*pi == k: that key is local only (each key once)
    (1, 3, 3, 25, 7, 30, 6, 2),     # band wider than N
    (1, 2, 2, 19, 3, 4, 100, 2),    # period beyond N: no skip key exists
    (1, 2, 2, 23, 4, 2, 5, 0),      # S = 0
]


@pytest.mark.parametrize("case", PI_CASES)
def test_pi_matches_dense_brute_force(case):
    B, H, Hkv, N, d, kl, per, S = case
    q, k, v, a = rand_case(B, H, Hkv, N, d, seed=N + d)
    out, lse, P = oracle.fwd(q, k, v, a, kl, per, S, 0, want_P=True)
    bo, bl, bP = dense_forward(q, k, v, a, kl, per, S, 0)
    np.testing.assert_allclose(out, bo.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, bl.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(P, bP.numpy(), atol=1e-12, rtol=0)


@pytest.mark.parametrize("N,c", [(50, 7), (48, 8), (20, 1), (16, 40), (33, 16)])
def test_ecp_matches_dense_brute_force(N, c):
    q, k, v, _ = rand_case(1, 2, 1, N, 6, seed=c)
    out, lse, P = oracle.fwd(q, k, v, None, c, 0, 0, 1, want_P=True)
    bo, bl, bP = dense_forward(q, k, v, None, c, 0, 0, 1)
    np.testing.assert_allclose(out, bo.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, bl.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(P, bP.numpy(), atol=1e-12, rtol=0)


def _sdpa(q, k, v, mask=None, causal=False):
    G = q.shape[1] // k.shape[1]
    kk = k.repeat_interleave(G, dim=1)
    vv = v.repeat_interleave(G, dim=1)
    return F.scaled_dot_product_attention(q, kk, vv, attn_mask=mask, is_causal=causal)


@pytest.mark.parametrize("kl", [0, 3, 16])
def test_s0_is_sliding_window_and_alpha_free(kl):
    """S=0: the prior is a per-row constant, so softmax removes it -> window attention."""
    N = 40
    q, k, v, a = rand_case(1, 4, 2, N, 8, seed=kl)
    i = torch.arange(N).view(N, 1)
    j = torch.arange(N).view(1, N)
    band = (i - j >= 0) & (i - j <= kl)
    ref = _sdpa(q, k, v, mask=band)
    out_a, _ = oracle.fwd(q, k, v, a, kl, 5, 0, 0)
    out_1, _ = oracle.fwd(q, k, v, torch.ones_like(a), kl, 5, 0, 0)
    np.testing.assert_allclose(out_a, ref.numpy(), atol=1e-12, rtol=0)
    np.testing.assert_allclose(out_1, ref.numpy(), atol=1e-12, rtol=0)


def test_wide_band_is_full_causal():
    N = 45
    q, k, v, a = rand_case(2, 2, 2, N, 8, seed=3)
    ref = _sdpa(q, k, v, causal=True)
    for kl in (N - 1, N + 10):
        out, _ = oracle.fwd(q, k, v, a, kl, 7, 0, 0)
        np.testing.assert_allclose(out, ref.numpy(), atol=1e-12, rtol=0)


@pytest.mark.parametrize("N,c", [(64, 16), (50, 9)])
def test_ecp_is_sdpa_with_block_mask(N, c):
    q, k, v, _ = rand_case(1, 4, 4, N, 8, seed=N)
    i = torch.arange(N).view(N, 1)
    j = torch.arange(N).view(1, N)
    s_i, s_j = i // c, j // c
    mask = (j <= i) & ((s_j == s_i) | (s_j == s_i - 1))
    ref = _sdpa(q, k, v, mask=mask)
    out, _ = oracle.fwd(q, k, v, None, c, 0, 0, 1)
    np.testing.assert_allclose(out, ref.numpy(), atol=1e-12, rtol=0)


def test_q_zero_closed_form():
    """q = 0: every score is 0, so weights are alpha on the band and 1-alpha on skips.

    out_i = (alpha_i sum_{L(i)} v_j + (1-alpha_i) sum_{P(i)} v_j)
            / (alpha_i |L(i)| + (1-alpha_i) |P(i)|)
    """
    B, H, N, d, kl, per, S = 1, 2, 60, 5, 6, 11, 4
    _, k, v, a = rand_case(B, H, H, N, d, seed=9)
    q = torch.zeros(B, H, N, d, dtype=torch.float64)
    out, lse = oracle.fwd(q, k, v, a, kl, per, S, 0)
    for h in range(H):
        for i in range(N):
            lo = max(0, i - kl)
            loc = v[0, h, lo:i + 1].sum(0)
            sk = [i - m * per for m in range(1, S + 1) if m * per > kl and i - m * per >= 0]
            skv = v[0, h, sk].sum(0) if sk else torch.zeros(d, dtype=torch.float64)
            al = float(a[0, h, i])
            den = al * (i - lo + 1) + (1 - al) * len(sk)
            exp_out = (al * loc + (1 - al) * skv) / den
            np.testing.assert_allclose(out[0, h, i], exp_out.numpy(), atol=1e-13, rtol=0)
            assert abs(lse[0, h, i] - math.log(den)) < 1e-13


def test_row_zero_special_case():
    """Row 0 sees only key 0 (local): out_0 = v_0, lse_0 = q0.k0/sqrt(d) + ln alpha_0."""
    q, k, v, a = rand_case(1, 3, 3, 20, 7, seed=21)
    out, lse = oracle.fwd(q, k, v, a, 4, 3, 3, 0)
    for h in range(3):
        np.testing.assert_allclose(out[0, h, 0], v[0, h, 0].numpy(), atol=1e-15, rtol=0)
        ref = float(q[0, h, 0] @ k[0, h, 0]) / math.sqrt(7) + math.log(float(a[0, h, 0]))
        assert abs(lse[0, h, 0] - ref) < 1e-13


def test_hand_worked_example():
    """N=3, d=2, k=0, pi=1, S=2, q=k=0, alpha=(1/2, 1/4, 1/2), v0=(1,0), v1=(0,1), v2=(1,1).

    Worked by hand from the definitions:
      row 0: L={0}, P={}      -> out=(1,0),            lse=ln(1/2)
      row 1: L={1}, P={0}     -> weights 1/4, 3/4     -> out=(3/4, 1/4), lse=ln(1)=0
      row 2: L={2}, P={1,0}   -> weights 1/2,1/2,1/2 over total 3/2
                              -> out=(2/3, 2/3),       lse=ln(3/2)
    """
    q = torch.zeros(1, 1, 3, 2, dtype=torch.float64)
    k = torch.zeros(1, 1, 3, 2, dtype=torch.float64)
    v = torch.tensor([[[[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]]]], dtype=torch.float64)
    a = torch.tensor([[[0.5, 0.25, 0.5]]], dtype=torch.float32)
    out, lse = oracle.fwd(q, k, v, a, 0, 1, 2, 0)
    np.testing.assert_allclose(out[0, 0], [[1, 0], [0.75, 0.25], [2 / 3, 2 / 3]], atol=1e-15)
    np.testing.assert_allclose(lse[0, 0], [math.log(0.5), 0.0, math.log(1.5)], atol=1e-15)


def test_hand_worked_example_with_scores():
    """N=2, d=1 (scale 1), k=1, S=0: row 1 has logits q1*k0 and q1*k1 (+ln alpha both).

    q1=1, k0=0, k1=ln 3 -> weights 1:3 -> out_1 = (v0 + 3 v1)/4, lse_1 = ln(4 alpha_1).
    """
    q = torch.tensor([[[[0.0], [1.0]]]], dtype=torch.float64)
    k = torch.tensor([[[[0.0], [math.log(3.0)]]]], dtype=torch.float64)
    v = torch.tensor([[[[2.0], [6.0]]]], dtype=torch.float64)
    a = torch.tensor([[[0.5, 0.5]]], dtype=torch.float32)
    out, lse = oracle.fwd(q, k, v, a, 1, 4, 0, 0)
    assert abs(out[0, 0, 1, 0] - (2.0 + 3 * 6.0) / 4) < 1e-14
    assert abs(lse[0, 0, 1] - math.log(4 * 0.5)) < 1e-14


@pytest.mark.parametrize("mode", [0, 1])
def test_rows_sum_to_one_and_zero_outside_union(mode):
    N = 70
    q, k, v, a = rand_case(1, 2, 2, N, 6, seed=5)
    kl, per, S = (9, 13, 4) if mode == 0 else (12, 0, 0)
    _, _, P = oracle.fwd(q, k, v, a if mode == 0 else None, kl, per, S, mode, want_P=True)
    np.testing.assert_allclose(P.sum(-1), 1.0, atol=1e-12, rtol=0)
    local, skip = union_masks(N, kl, per, S, mode)
    outside = ~(local | skip).numpy()
    assert np.all(P[..., outside] == 0.0)
    assert np.all(P[..., ~outside] > 0.0)


def test_gqa_equals_repeated_heads():
    B, H, Hkv, N, d = 1, 8, 2, 40, 6
    q, k, v, a = rand_case(B, H, Hkv, N, d, seed=17)
    out_g, lse_g = oracle.fwd(q, k, v, a, 5, 8, 3, 0)
    G = H // Hkv
    out_r, lse_r = oracle.fwd(q, k.repeat_interleave(G, 1), v.repeat_interleave(G, 1), a, 5, 8, 3, 0)
    np.testing.assert_array_equal(out_g, out_r)
    np.testing.assert_array_equal(lse_g, lse_r)


def test_bf16_bits_read_exactly():
    q, k, v, a = rand_case(1, 2, 2, 30, 16, seed=2)
    qb, kb, vb = q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)
    o1, l1 = oracle.fwd(qb, kb, vb, a, 4, 6, 2, 0)
    o2, l2 = oracle.fwd(qb.double(), kb.double(), vb.double(), a, 4, 6, 2, 0)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_row_range_equals_full():
    q, k, v, a = rand_case(2, 2, 1, 50, 4, seed=8)
    out, lse = oracle.fwd(q, k, v, a, 6, 10, 3, 0)
    o2, l2 = oracle.fwd(q, k, v, a, 6, 10, 3, 0, rows=(17, 44))
    np.testing.assert_array_equal(o2, out[:, :, 17:44])
    np.testing.assert_array_equal(l2, lse[:, :, 17:44])


def test_alpha_edges():
    """alpha=0 removes the band (row 0 has no skip -> out 0, lse -inf); alpha=1 removes skips."""
    N, kl, per, S = 30, 3, 8, 2
    q, k, v, _ = rand_case(1, 1, 1, N, 4, seed=4)
    a0 = torch.zeros(1, 1, N)
    out0, lse0 = oracle.fwd(q, k, v, a0, kl, per, S, 0)
    for i in range(N):
        sk = [i - m * per for m in range(1, S + 1) if m * per > kl and i - m * per >= 0]
        if not sk:
            assert lse0[0, 0, i] == -np.inf and np.all(out0[0, 0, i] == 0.0)
        else:
            z = np.array([float(q[0, 0, i] @ k[0, 0, j]) / 2.0 for j in sk])
            w = np.exp(z - z.max()) / np.exp(z - z.max()).sum()
            ref = (w[:, None] * v[0, 0, sk].numpy()).sum(0)
            np.testing.assert_allclose(out0[0, 0, i], ref, atol=1e-13)
    a1 = torch.ones(1, 1, N)
    out1, _ = oracle.fwd(q, k, v, a1, kl, per, S, 0)
    out_band, _ = oracle.fwd(q, k, v, a1, kl, per, 0, 0)
    np.testing.assert_allclose(out1, out_band, atol=1e-15)


# --------------------------------------------------------------------------- counts

def closed_form_counts(N, kl, per, S, mode):
    """Per-row neighbour count and key-index sum from closed forms (numpy, vectorised)."""
    i = np.arange(N, dtype=np.int64)
    if mode == 0:
        lo = np.maximum(0, i - kl)
    else:
        lo = np.maximum(0, (i // kl - 1) * kl)
    cnt = i - lo + 1
    isum = (lo + i) * (i - lo + 1) // 2
    if mode == 0:
        for m in range(1, S + 1):
            back = m * per
            if back <= kl:
                continue
            ok = i - back >= 0
            cnt = cnt + ok
            isum = isum + np.where(ok, i - back, 0)
    return cnt, isum


def closed_form_total(N, kl, per, S, mode):
    """Attended pairs per (b, h): band N(k+1) - k(k+1)/2 (k < N), skip sum max(0, N - m pi);
    ECP per half-segment s>=1 of length n_s: n_s (c+1) + n_s (n_s - 1)/2, segment 0: n0(n0+1)/2."""
    if mode == 0:
        band = N * (kl + 1) - kl * (kl + 1) // 2 if kl < N else N * (N + 1) // 2
        skip = sum(max(0, N - m * per) for m in range(1, S + 1) if m * per > kl)
        return band + skip
    if mode == 2:  # bidirectional: every offset 0 < t <= k twice, the diagonal once
        from tests.test_oracle_pins_bidir import closed_form_total as bidir_total
        return bidir_total(N, kl, per, S)
    c = kl
    total, s = 0, 0
    while s * c < N:
        n = min(c, N - s * c)
        total += n * (n + 1) // 2 if s == 0 else n * (c + 1) + n * (n - 1) // 2
        s += 1
    return total


COUNT_CASES = [
    (256, 16, 32, 1, 0), (4096, 128, 256, 1, 0), (8192, 512, 0, 0, 1),
    (65536, 256, 1024, 4, 0), (16384, 256, 512, 2, 0),
    (100, 10, 4, 5, 0), (77, 5, 3, 0, 0), (90, 12, 6, 4, 0), (1000, 37, 0, 0, 1), (50, 60, 10, 3, 0),
]


@pytest.mark.parametrize("case", COUNT_CASES)
def test_counts_closed_forms(case):
    N, kl, per, S, mode = case
    cnt, isum = oracle.counts(N, kl, per, S, mode)
    c2, s2 = closed_form_counts(N, kl, per, S, mode)
    np.testing.assert_array_equal(cnt, c2)
    np.testing.assert_array_equal(isum, s2)
    assert int(cnt.sum()) == closed_form_total(N, kl, per, S, mode)


def test_golden_pair_counts():
    """Per-(b,h) attended-pair totals of the workloads (tests/golden/pair_counts.json)."""
    with open(os.path.join(GOLDEN, "pair_counts.json")) as f:
        gold = json.load(f)
    for name, rec in gold["workloads"].items():
        cnt, isum = oracle.counts(rec["N"], rec["k_local"], rec["period"], rec["S"], rec["mode"])
        assert int(cnt.sum()) == rec["pairs_per_head"], name
        assert int(isum.sum()) == rec["index_sum_per_head"], name
        assert closed_form_total(rec["N"], rec["k_local"], rec["period"], rec["S"],
                                 rec["mode"]) == rec["pairs_per_head"], name


# --------------------------------------------------------------------------- backward

def _loss(q, k, v, a, dout, kl, per, S, mode):
    out, _ = oracle.fwd(q, k, v, a, kl, per, S, mode)
    return float((out * dout.numpy()).sum())


@pytest.mark.parametrize("mode", [0, 1])
def test_bwd_finite_differences(mode):
    B, H, Hkv, N, d = 1, 2, 1, 14, 3
    kl, per, S = (2, 4, 3) if mode == 0 else (4, 0, 0)
    q, k, v, a = rand_case(B, H, Hkv, N, d, seed=31, alpha_lo=0.2, alpha_hi=0.8)
    a = a.double()
    g = torch.Generator().manual_seed(5)
    dout = torch.randn(B, H, N, d, generator=g, dtype=torch.float64)
    am = a if mode == 0 else None
    dq, dk, dv, dal = oracle.bwd(q, k, v, am.float() if am is not None else None, dout,
                                 kl, per, S, mode)
    eps = 1e-6

    def fd(t, idx, alpha_t=None):
        t2p, t2m = t.clone(), t.clone()
        t2p[idx] += eps
        t2m[idx] -= eps
        return t2p, t2m

    rng = np.random.default_rng(0)
    for name, t, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, s)) for s in t.shape)
            tp, tm = fd(t, idx)
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = tp, tm
            lp = _loss(args_p["q"], args_p["k"], args_p["v"], am, dout, kl, per, S, mode)
            lm = _loss(args_m["q"], args_m["k"], args_m["v"], am, dout, kl, per, S, mode)
            num = (lp - lm) / (2 * eps)
            assert abs(num - grad[idx]) <= 1e-6 * max(1.0, abs(num)), (name, idx, num, grad[idx])
    if mode == 0:
        # alpha is read as fp32 by the oracle, so difference it in fp64 through the dense form
        for _ in range(6):
            idx = tuple(int(rng.integers(0, s)) for s in a.shape)
            ap, amn = a.clone(), a.clone()
            ap[idx] += 1e-5
            amn[idx] -= 1e-5
            op, _, _ = dense_forward(q, k, v, ap, kl, per, S, 0)
            om, _, _ = dense_forward(q, k, v, amn, kl, per, S, 0)
            num = float(((op - om) * dout).sum()) / 2e-5
            # oracle dalpha is at the fp32-rounded alpha; compare loosely against fp64 alpha
            assert abs(num - dal[idx]) <= 1e-4 * max(1.0, abs(num)), (idx, num, dal[idx])


@pytest.mark.parametrize("case", [(1, 4, 2, 29, 5, 4, 6, 3, 0), (2, 2, 2, 31, 4, 7, 0, 0, 1),
                                  (1, 2, 1, 26, 6, 10, 4, 4, 0)])
def test_bwd_matches_autograd_through_brute_force(case):
    B, H, Hkv, N, d, kl, per, S, mode = case
    q, k, v, a = rand_case(B, H, Hkv, N, d, seed=N, alpha_lo=0.1, alpha_hi=0.9)
    g = torch.Generator().manual_seed(1)
    dout = torch.randn(B, H, N, d, generator=g, dtype=torch.float64)
    am = a if mode == 0 else None
    dq, dk, dv, dal = oracle.bwd(q, k, v, am, dout, kl, per, S, mode)
    qt, kt, vt = (t.clone().requires_grad_(True) for t in (q, k, v))
    at = a.double().clone().requires_grad_(True) if mode == 0 else None
    out, _, _ = dense_forward(qt, kt, vt, at, kl, per, S, mode)
    out.backward(dout)
    np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-10, rtol=0)
    np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-10, rtol=0)
    np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-10, rtol=0)
    if mode == 0:
        np.testing.assert_allclose(dal, at.grad.numpy(), atol=1e-9, rtol=1e-9)
    else:
        assert np.all(dal == 0.0)


def test_dalpha_skip_only_form_and_zero_without_skips():
    """sum_j dz_ij = 0 (softmax rows), so dalpha_i = -sum_{P(i)} dz_ij / (alpha_i (1 - alpha_i)).

    Checked through autograd on the dense form: the gradient of the loss with respect to
    the skip-logit bias equals sum_{P(i)} dz_ij.  Without skip keys dalpha is 0.
    """
    B, H, N, d, kl, per, S = 1, 2, 40, 5, 4, 9, 3
    q, k, v, a = rand_case(B, H, H, N, d, seed=77, alpha_lo=0.2, alpha_hi=0.8)
    g = torch.Generator().manual_seed(3)
    dout = torch.randn(B, H, N, d, generator=g, dtype=torch.float64)
    _, _, _, dal = oracle.bwd(q, k, v, a, dout, kl, per, S, 0)
    # dense: separate the local and skip biases as leaves
    local, skip = union_masks(N, kl, per, S, 0)
    scores = (q @ k.transpose(-1, -2)) / math.sqrt(d)
    ad = a.double()
    bl = torch.log(ad).unsqueeze(-1).expand(B, H, N, N).clone().requires_grad_(True)
    bs = torch.log1p(-ad).unsqueeze(-1).expand(B, H, N, N).clone().requires_grad_(True)
    z = torch.where(local, scores + bl, torch.where(skip, scores + bs, torch.tensor(-math.inf,
                                                                                   dtype=torch.float64)))
    out = torch.softmax(z, -1) @ v
    out.backward(dout)
    sum_skip = (bs.grad * skip).sum(-1)
    sum_local = (bl.grad * local).sum(-1)
    np.testing.assert_allclose((sum_local + sum_skip).numpy(), 0.0, atol=1e-11)
    ref = -sum_skip / (ad * (1 - ad))
    np.testing.assert_allclose(dal, ref.numpy(), atol=1e-9, rtol=1e-9)
    _, _, _, dal0 = oracle.bwd(q, k, v, a, dout, kl, per, 0, 0)
    np.testing.assert_allclose(dal0, 0.0, atol=1e-12)


def test_dalpha_at_a_saturated_gate_is_zero_and_the_rest_unchanged():
    """At alpha exactly 0 or 1 one prior is -inf and its weights are exactly 0; the oracle takes
    dalpha there as 0 (a saturated gate passes no gradient) instead of 0/0.  Every other row keeps
    the chain-rule value, and dq, dk, dv still match autograd through the dense form."""
    B, H, N, d, kl, per, S = 1, 2, 40, 5, 4, 9, 3
    q, k, v, a = rand_case(B, H, H, N, d, seed=78, alpha_lo=0.2, alpha_hi=0.8)
    g = torch.Generator().manual_seed(4)
    dout = torch.randn(B, H, N, d, generator=g, dtype=torch.float64)
    a_sat = a.clone()
    a_sat[:, 0, ::3] = 0.0
    a_sat[:, 1, 1::4] = 1.0
    sat = ((a_sat == 0.0) | (a_sat == 1.0)).numpy()
    dq, dk, dv, dal = oracle.bwd(q, k, v, a_sat, dout, kl, per, S, 0)
    assert np.all(np.isfinite(dal)) and np.all(dal[sat] == 0.0)
    _, _, _, dal_ref = oracle.bwd(q, k, v, a, dout, kl, per, S, 0)
    # rows whose gate did not change keep their value (each row's dalpha depends on that row only)
    unchanged = (a_sat == a).numpy()
    np.testing.assert_allclose(dal[unchanged], dal_ref[unchanged], rtol=1e-12, atol=0)
    # dense reference with the union masks; rows with alpha = 0 and no skip key have no finite
    # logit: their output is 0 and they pass no gradient
    qt, kt, vt = (t.clone().requires_grad_(True) for t in (q, k, v))
    local, skip = union_masks(N, kl, per, S, 0)
    ad = a_sat.double().unsqueeze(-1)
    scores = (qt @ kt.transpose(-1, -2)) / math.sqrt(d)
    ninf = torch.tensor(-math.inf, dtype=torch.float64)
    z = torch.where(local, scores + torch.log(ad), torch.where(skip, scores + torch.log1p(-ad), ninf))
    dead = torch.isinf(z).all(-1, keepdim=True)
    p_ = torch.softmax(torch.where(dead, torch.zeros_like(z), z), -1)
    out = (p_ @ vt) * (~dead)
    out.backward(dout)
    np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-10, rtol=0)
    np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-10, rtol=0)
    np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-10, rtol=0)
