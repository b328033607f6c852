"""Pins for the oracle's gate: a per-head MLP of one hidden layer on the head's query,
hid_f = max(0, W1_h[f] . q + b1_h[f]) and alpha = 1 / (1 + exp(-(w2_h . hid + b2_h))).

"pi-Attention: Periodic Sparse Transformers for Efficient Long-Context Modeling", section 2.3:
a light neural network (MLP) produces alpha per token and per head from the input content, and
alpha enters the one softmax over the union as a log-prior (+ln alpha on band logits,
+ln(1 - alpha) on skip logits).  The pins tie the gate to values the mathematics fixes: exact
values of the logistic function (1/2, 3/4, 1/4, 9/10), a hand-worked network in which the ReLU
switches units off, the symmetry alpha(-z) = 1 - alpha(z), and saturated gates, which reduce the
gated attention to library attention with independently built masks.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

PI, BIDIR = 0, 2
HID = 8  # hidden units per head


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


def zeros(H, d):
    return (torch.zeros(H, HID, d, dtype=torch.float64), torch.zeros(H, HID, dtype=torch.float64),
            torch.zeros(H, HID, dtype=torch.float64), torch.zeros(H, dtype=torch.float64))


def test_zero_hidden_layer_gives_the_logistic_of_the_output_bias():
    """W1 = 0 and b1 = 0 switch every hidden unit off, so alpha = 1 / (1 + exp(-b2_h)); the
    logistic function takes the exact values 1/2, 3/4, 1/4 and 9/10 at 0, ln 3, -ln 3, ln 9."""
    H, d = 4, 16
    w1, b1, w2, b2 = zeros(H, d)
    w2[:] = 7.0  # unused: no unit is on
    b2[:] = torch.tensor([0.0, math.log(3.0), -math.log(3.0), math.log(9.0)], dtype=torch.float64)
    q = torch.randn(2, H, 5, d, dtype=torch.float64)
    alpha = oracle.gate(q, w1, b1, w2, b2)
    for h, want in enumerate((0.5, 0.75, 0.25, 0.9)):
        np.testing.assert_allclose(alpha[:, h], want, rtol=0, atol=2e-16)


def test_hand_worked_network():
    """d = 4, q = (1, -2, 1/2, 3).  Unit 0 reads q_0 with bias 1/2: 3/2.  Unit 1 reads q_1: -2,
    switched off by the ReLU (its output weight 5 must not count).  Unit 2 reads 2 q_2: 1.  Unit
    3 reads q_3 - q_0 with bias -1: 1.  Units 4-7 have bias -1 and no input: off.  With output
    weights (1, 5, 2, -1/2, 9, 9, 9, 9) the logit is 3/2 + 2 - 1/2 = 3, and b2 = ln 3 - 3 gives
    z = ln 3, alpha = 3/4.  Reading the weights transposed ([d, F]), dropping b1, skipping the ReLU
    or scaling the logit would each move alpha away from 3/4."""
    H, d = 1, 4
    w1, b1, w2, b2 = zeros(H, d)
    w1[0, 0, 0] = 1.0
    b1[0, 0] = 0.5
    w1[0, 1, 1] = 1.0
    w1[0, 2, 2] = 2.0
    w1[0, 3, 3], w1[0, 3, 0] = 1.0, -1.0
    b1[0, 3] = -1.0
    b1[0, 4:] = -1.0
    w2[0] = torch.tensor([1.0, 5.0, 2.0, -0.5, 9.0, 9.0, 9.0, 9.0], dtype=torch.float64)
    b2[0] = math.log(3.0) - 3.0
    q = torch.tensor([1.0, -2.0, 0.5, 3.0], dtype=torch.float64).view(1, 1, 1, d)
    alpha = oracle.gate(q, w1, b1, w2, b2)
    np.testing.assert_allclose(alpha[0, 0, 0], 0.75, rtol=0, atol=1e-15)


def test_output_sign_flip_gives_one_minus_alpha():
    """The logistic function is odd about 1/2: negating w2 and b2 maps alpha to 1 - alpha."""
    H, d = 3, 32
    g = torch.Generator().manual_seed(5)
    w1 = torch.randn(H, HID, d, generator=g, dtype=torch.float64) / math.sqrt(d)
    b1 = torch.randn(H, HID, generator=g, dtype=torch.float64)
    w2 = torch.randn(H, HID, generator=g, dtype=torch.float64)
    b2 = torch.randn(H, generator=g, dtype=torch.float64)
    q = torch.randn(2, H, 9, d, generator=g, dtype=torch.float64)
    a = oracle.gate(q, w1, b1, w2, b2)
    a_neg = oracle.gate(q, w1, b1, -w2, -b2)
    np.testing.assert_allclose(a + a_neg, 1.0, rtol=0, atol=1e-15)
    assert np.all((a > 0.0) & (a < 1.0)) and np.std(a) > 0.05


@pytest.mark.parametrize("mode", [PI, BIDIR])
def test_saturated_gates_reduce_to_library_attention(mode):
    """b2 = +/-60 with the hidden layer off: alpha -> 1 leaves the band alone, alpha -> 0 the skip
    keys alone (the band where a row has none), b2 = 0 the plain union."""
    B, H, Hkv, N, d, kl, per, S = 1, 4, 2, 70, 8, 5, 16, 3
    q, k, v = case(B, H, Hkv, N, d, seed=3 + mode)
    w1, b1, w2, b2 = zeros(H, d)
    b2[:] = torch.tensor([60.0, -60.0, 0.0, 60.0], dtype=torch.float64)
    out, lse, alpha = oracle.fwd_gated(q, k, v, (w1, b1, w2, b2), kl, per, S, mode)
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
    """One hidden unit reads q_0 with weight 1; its output weight is +80 on head 0 and -80 on
    head 1, with b2 = -40 / +40.  A row with q_0 = +1 then has z = +40 (head 0) or -40 (head 1),
    a row with q_0 = -1 has the unit off and z = -40 / +40: each row is switched between the
    band-only and the skip-dominated attention by its own query and its own head's weights; the
    other query components do not enter the gate."""
    B, H, Hkv, N, d, kl, per, S = 2, 2, 1, 60, 6, 4, 12, 3
    q, k, v = case(B, H, Hkv, N, d, seed=11)
    g = torch.Generator().manual_seed(12)
    sign = torch.where(torch.rand(B, H, N, generator=g) < 0.5, -1.0, 1.0).double()
    q[..., 0] = sign
    w1, b1, w2, b2 = zeros(H, d)
    w1[:, 0, 0] = 1.0
    w2[0, 0], w2[1, 0] = 80.0, -80.0
    b2[0], b2[1] = -40.0, 40.0
    out, _, alpha = oracle.fwd_gated(q, k, v, (w1, b1, w2, b2), kl, per, S, PI)
    band, skip = masks(N, kl, per, S, PI)
    has_skip = skip.any(dim=1)
    ref_band = sdpa(q, k, v, band).numpy()
    ref_skip = sdpa(q, k, v, torch.where(has_skip.view(N, 1), skip, band)).numpy()
    for b in range(B):
        for h in range(H):
            for i in range(N):
                on = float(sign[b, h, i]) > 0
                band_side = (on and h == 0) or (not on and h == 1)  # alpha -> 1
                ref = ref_band if band_side else ref_skip
                np.testing.assert_allclose(out[b, h, i], ref[b, h, i], atol=1e-10, rtol=0)
                assert (alpha[b, h, i] > 0.5) == band_side


def test_gate_on_bf16_queries_uses_their_exact_values():
    """bf16 queries enter the gate with their exact values: the bf16 and the widened fp64
    tensors give the same alpha."""
    q = torch.randn(1, 3, 17, 64, dtype=torch.float32).bfloat16()
    g = torch.Generator().manual_seed(2)
    w1 = torch.randn(3, HID, 64, generator=g, dtype=torch.float64) * 0.1
    b1 = torch.randn(3, HID, generator=g, dtype=torch.float64)
    w2 = torch.randn(3, HID, generator=g, dtype=torch.float64)
    b2 = torch.randn(3, generator=g, dtype=torch.float64)
    a16 = oracle.gate(q, w1, b1, w2, b2)
    a64 = oracle.gate(q.double(), w1, b1, w2, b2)
    np.testing.assert_array_equal(a16, a64)
