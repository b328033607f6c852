"""Pins for the oracle's gate: alpha = 1 / (1 + exp(-(q . w_h + c_h))) per query row and head.

"pi-Attention: Periodic Sparse Transformers for Efficient Long-Context Modeling", section 2.3:
a light per-token, per-head network produces alpha from the input content, and alpha enters the
one softmax over the union as a log-prior (+ln alpha on band logits, +ln(1 - alpha) on skip
logits).  The network's form is not given; the oracle takes a one-layer logistic gate on the
head's query.  Saturated gates reduce the gated attention to library attention with an
independently built mask: alpha -> 1 leaves the band alone, alpha -> 0 the skip keys alone (the
band where a row has none), alpha = 1/2 the plain union.  A gate switched per row by the sign of
one query component pins which component and which head's weights the gate reads.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

PI, BIDIR = 0, 2


def masks(N, kl, per, S, mode):
    """Boolean band and skip masks [N, N] from broadcast index arithmetic."""
    i = torch.arange(N).view(N, 1)
    j = torch.arange(N).view(1, N)
    if mode == BIDIR:
        band = (j - i).abs() <= kl
    else:
        band = (j <= i) & (j >= i - kl)
    skip = torch.zeros(N, N, dtype=torch.bool)
    for m in range(1, S + 1):
        if m * per <= kl:
            continue
        skip |= j == i - m * per
        if mode == BIDIR:
            skip |= j == i + m * per
    return band, skip


def sdpa(q, k, v, mask):
    G = q.shape[1] // k.shape[1]
    return F.scaled_dot_product_attention(q, k.repeat_interleave(G, 1), v.repeat_interleave(G, 1),
                                          attn_mask=mask)


def case(B, H, Hkv, N, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, N, d, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float64)
    return q, k, v


@pytest.mark.parametrize("mode", [PI, BIDIR])
def test_saturated_gates_reduce_to_library_attention(mode):
    B, H, Hkv, N, d, kl, per, S = 1, 4, 2, 70, 8, 5, 16, 3
    q, k, v = case(B, H, Hkv, N, d, seed=3 + mode)
    w = torch.zeros(H, d, dtype=torch.float64)
    c = torch.tensor([60.0, -60.0, 0.0, 60.0], dtype=torch.float64)
    out, lse, alpha = oracle.fwd_gated(q, k, v, w, c, kl, per, S, mode)
    band, skip = masks(N, kl, per, S, mode)
    has_skip = skip.any(dim=1)
    ref_band = sdpa(q, k, v, band).numpy()
    ref_union = sdpa(q, k, v, band | skip).numpy()
    skip_or_band = torch.where(has_skip.view(N, 1), skip, band)
    ref_skip = sdpa(q, k, v, skip_or_band).numpy()
    for h, ref in ((0, ref_band), (1, ref_skip), (2, ref_union), (3, ref_band)):
        np.testing.assert_allclose(out[0, h], ref[0, h], atol=1e-10, rtol=0)
    np.testing.assert_allclose(alpha[0, 2], 0.5, atol=0, rtol=0)


def test_gate_reads_its_head_weights_and_the_rows_query():
    """w_h = (+/-80, 0, ...) and q[..., 0] = +/-1 switch each row between the band-only and
    the skip-dominated attention; the other query components do not enter the gate."""
    B, H, Hkv, N, d, kl, per, S = 2, 2, 1, 60, 6, 4, 12, 3
    q, k, v = case(B, H, Hkv, N, d, seed=11)
    g = torch.Generator().manual_seed(12)
    sign = torch.where(torch.rand(B, H, N, generator=g) < 0.5, -1.0, 1.0).double()
    q[..., 0] = sign
    w = torch.zeros(H, d, dtype=torch.float64)
    w[0, 0], w[1, 0] = 80.0, -80.0
    c = torch.zeros(H, dtype=torch.float64)
    out, _, alpha = oracle.fwd_gated(q, k, v, w, c, kl, per, S, PI)
    band, skip = masks(N, kl, per, S, PI)
    has_skip = skip.any(dim=1)
    ref_band = sdpa(q, k, v, band).numpy()
    ref_skip = sdpa(q, k, v, torch.where(has_skip.view(N, 1), skip, band)).numpy()
    for b in range(B):
        for h in range(H):
            for i in range(N):
                band_side = float(sign[b, h, i]) * float(w[h, 0]) > 0  # alpha -> 1
                ref = ref_band if band_side else ref_skip
                np.testing.assert_allclose(out[b, h, i], ref[b, h, i], atol=1e-10, rtol=0)
                assert (alpha[b, h, i] > 0.5) == band_side


def test_gate_on_bf16_queries_uses_their_exact_values():
    """bf16 queries enter the gate with their exact values: the bf16 and the widened fp64
    tensors give the same alpha."""
    q = torch.randn(1, 3, 17, 64, dtype=torch.float32).bfloat16()
    w = torch.randn(3, 64, dtype=torch.float64) * 0.1
    c = torch.randn(3, dtype=torch.float64)
    a16 = oracle.gate(q, w, c)
    a64 = oracle.gate(q.double(), w, c)
    np.testing.assert_array_equal(a16, a64)
