"""Dense brute-force pi-Attention / ECP attention in torch fp64 (a pin for the oracle).

This is deliberately a *different* formulation from the oracle: the neighbour
set is a broadcast boolean mask over the full N x N score matrix (built from
the position difference i - j and from half-segment numbers), the prior is a
dense bias matrix, and the softmax is torch's.  It is differentiable, so torch
autograd gives an independent backward.  Tiny N only.

Definitions follow "pi-Attention: Periodic Sparse Transformers for Efficient
Long-Context Modeling" section 2.1-2.3 and the ECP page, section 2 (PAR block).
"""
import math

import torch


def union_masks(N, k_local, period, S, mode):
    """(local, skip) boolean [N, N] masks; for ECP skip is all False.  Mode 2 is the
    bidirectional form of the band and skips (same page, 2.1 and 2.2)."""
    i = torch.arange(N).view(N, 1)
    j = torch.arange(N).view(1, N)
    diff = i - j
    if mode == 0:
        local = (diff >= 0) & (diff <= k_local)
        skip = torch.zeros(N, N, dtype=torch.bool)
        for m in range(1, S + 1):
            if m * period > k_local:
                skip |= diff == m * period
    elif mode == 2:  # bidirectional: |i - j| <= k, skips at i -/+ m*period
        local = diff.abs() <= k_local
        skip = torch.zeros(N, N, dtype=torch.bool)
        for m in range(1, S + 1):
            if m * period > k_local:
                skip |= diff.abs() == m * period
    else:
        c = k_local
        local = (diff >= 0) & ((j // c) >= (i // c) - 1)
        skip = torch.zeros(N, N, dtype=torch.bool)
    return local, skip


def dense_forward(q, k, v, alpha, k_local, period, S, mode):
    """q [B,H,N,d], k/v [B,Hkv,N,d] fp64 torch tensors; alpha [B,H,N] or None.

    Returns (out, lse, P) with P the dense [B,H,N,N] probabilities.
    """
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    G = H // Hkv
    kk = k.repeat_interleave(G, dim=1)
    vv = v.repeat_interleave(G, dim=1)
    local, skip = union_masks(N, k_local, period, S, mode)
    scores = torch.matmul(q, kk.transpose(-1, -2)) / math.sqrt(d)
    neg_inf = torch.tensor(float("-inf"), dtype=q.dtype)
    if mode in (0, 2):
        a = alpha.to(q.dtype).unsqueeze(-1) if alpha is not None else torch.ones(B, H, N, 1,
                                                                                dtype=q.dtype)
        bias = torch.where(local, torch.log(a), torch.where(skip, torch.log1p(-a), neg_inf))
    else:
        bias = torch.where(local, torch.zeros((), dtype=q.dtype), neg_inf).expand(B, H, N, N)
    z = scores + bias
    lse = torch.logsumexp(z, dim=-1)
    finite = torch.isfinite(lse)
    safe = torch.where(finite, lse, torch.zeros_like(lse))
    P = torch.where(finite.unsqueeze(-1), torch.exp(z - safe.unsqueeze(-1)), torch.zeros_like(z))
    out = torch.matmul(P, vv)
    return out, lse, P
