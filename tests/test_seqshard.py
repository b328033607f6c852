"""Sequence sharding: the halo plan (host logic) and its exchange on world-size-2 gloo ranks (CPU).

The plan is checked against neighbour sets enumerated query by query from the definition
("pi-Attention" page, 2.1 band and 2.2 skips in the causal and the general bidirectional form;
ECP page, section 2, previous half-segment).  The exchange is checked end to end: two gloo
ranks each hold their own rows, exchange halos, attend on their local windows and return the
gradients of the halo rows to their owners; the concatenated shard results must equal the
whole-sequence oracle.  On the CPU the per-shard attention is the oracle on the shard's window
(the tests pass it in; the library's kernels need a GPU and are checked against the same plan
in test_gpu_seqshard.py).
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from structured_sparse_long_gb300 import seqshard as ss

PI, ECP, BIDIR = 0, 1, 2


def brute_keys(i, N, k, per, S, mode):
    """Keys of query i, one by one from the definition."""
    if mode == ECP:
        return set(range(max(0, (i // k - 1) * k), i + 1))
    keys = {j for j in range(N) if (i - k <= j <= i) or (mode == BIDIR and i <= j <= i + k)}
    for m in range(1, S + 1):
        if m * per > k:
            for j in (i - m * per, i + m * per) if mode == BIDIR else (i - m * per,):
                if 0 <= j < N:
                    keys.add(j)
    return keys


PLANS = [
    (1000, 2, 40, 300, 2, PI), (1000, 3, 40, 300, 2, BIDIR), (1000, 3, 100, 0, 0, ECP),
    (700, 4, 16, 64, 3, PI), (4096, 4, 256, 1024, 4, PI), (4096, 3, 256, 1024, 4, BIDIR),
    (2048, 2, 512, 0, 0, ECP), (600, 2, 8, 200, 5, PI), (513, 3, 20, 7, 9, BIDIR),
    (640, 5, 50, 40, 2, PI),  # band longer than the first skip: m = 1 is in the band
]


@pytest.mark.parametrize("N,world,k,per,S,mode", PLANS)
def test_plan_moves_exactly_the_halo(N, world, k, per, S, mode):
    """Every key of every shard query lies in the shard's window; the rows received are exactly
    the attended keys the shard does not own, each from its owner; sends mirror receives; the
    window starts where the kernels' blocks (and ECP's segments) stay aligned."""
    plans = ss.plan(N, world, k, per, S, mode)
    assert [p.t0 for p in plans][0] == 0 and plans[-1].t1 == N
    for a, b in zip(plans, plans[1:]):
        assert a.t1 == b.t0 and a.t1 % 128 == 0
    for p in plans:
        need = set()
        for i in range(p.t0, p.t1):
            need |= brute_keys(i, N, k, per, S, mode)
        assert min(need) >= p.w0 and max(need) < p.w1
        got = set()
        for pc in p.recv:
            t0, t1 = plans[pc.peer].t0, plans[pc.peer].t1
            assert t0 <= pc.a < pc.b <= t1 and pc.peer != p.rank
            rows = set(range(pc.a, pc.b))
            assert not (rows & got)
            got |= rows
            assert ss.Piece(p.rank, pc.a, pc.b) in plans[pc.peer].send
        assert got == need - set(range(p.t0, p.t1))
        assert ss.halo_rows(p) == len(got)
        assert p.q_offset % 128 == 0 and p.q_offset >= 0 and p.w1 <= N
        if mode == ECP:
            assert p.w0 % k == 0
    n_send = sum(len(p.send) for p in plans)
    assert n_send == sum(len(p.recv) for p in plans)


def test_split_rejects_too_many_shards():
    with pytest.raises(ValueError):
        ss.split(300, 4)


# ---------------------------------------------------------------- two gloo ranks

def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


CASES = [  # (B, H, Hkv, N, d, k, per, S, mode)
    (1, 4, 2, 600, 16, 24, 100, 3, PI),
    (2, 2, 1, 520, 8, 30, 150, 2, BIDIR),
    (1, 2, 2, 700, 8, 100, 0, 0, ECP),
]


def _inputs(case, seed):
    B, H, Hkv, N, d = case[:5]
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, N, d, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, N, d, generator=g, dtype=torch.float64)
    alpha = torch.sigmoid(torch.randn(B, H, N, generator=g)).float()
    dout = torch.randn(B, H, N, d, generator=g, dtype=torch.float64)
    return q, k, v, alpha, dout


def _embed(x, q_offset, n_win, fill):
    """Rows of the shard's queries placed at their key rows of the window."""
    shape = list(x.shape)
    shape[2] = n_win
    full = torch.full(shape, fill, dtype=x.dtype)
    full[:, :, q_offset:q_offset + x.shape[2]] = x
    return full


def _oracle_fwd_shard(q, k_win, v_win, alpha, q_offset, k_local, period, S, mode):
    import oracle
    n, nw = q.shape[2], k_win.shape[2]
    out, lse = oracle.fwd(_embed(q, q_offset, nw, 0.0), k_win, v_win, _embed(alpha, q_offset, nw, 0.5),
                          k_local, period, S, mode, rows=(q_offset, q_offset + n))
    return torch.from_numpy(out), torch.from_numpy(lse)


def _oracle_bwd_shard(q, k_win, v_win, alpha, out, lse, dout, q_offset, k_local, period, S, mode):
    """The window's rows of the gradient with the shard's queries only: the other rows of the
    window carry zero dout, so they add nothing to dk and dv."""
    import oracle
    n, nw = q.shape[2], k_win.shape[2]
    dq, dk, dv, dal = oracle.bwd(_embed(q, q_offset, nw, 0.0), k_win, v_win,
                                 _embed(alpha, q_offset, nw, 0.5), _embed(dout, q_offset, nw, 0.0),
                                 k_local, period, S, mode)
    sl = slice(q_offset, q_offset + n)
    return (torch.from_numpy(dq[:, :, sl]), torch.from_numpy(dk), torch.from_numpy(dv),
            torch.from_numpy(dal[:, :, sl]))


def _worker(rank, world, port, queue):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        res = []
        for ci, case in enumerate(CASES):
            B, H, Hkv, N, d, k, per, S, mode = case
            q, kk, v, alpha, dout = _inputs(case, seed=100 + ci)
            p = ss.plan(N, world, k, per, S, mode)[rank]
            own = slice(p.t0, p.t1)
            out, lse, ctx = ss.forward(q[:, :, own], kk[:, :, own], v[:, :, own], alpha[:, :, own], p,
                                       k, per, S, mode, attend=_oracle_fwd_shard)
            dq, dk, dv, dal = ss.backward(ctx, dout[:, :, own].contiguous(), attend_bwd=_oracle_bwd_shard)
            res.append(tuple(t.numpy() for t in (out, lse, dq, dk, dv, dal)))
        queue.put((rank, res))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_match_the_whole_sequence_oracle():
    import oracle
    oracle.build()  # once, before the ranks start
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(queue.get(timeout=300) for _ in range(2))
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    for ci, case in enumerate(CASES):
        B, H, Hkv, N, d, k, per, S, mode = case
        q, kk, v, alpha, dout = _inputs(case, seed=100 + ci)
        out, lse = oracle.fwd(q, kk, v, alpha, k, per, S, mode)
        dq, dk, dv, dal = oracle.bwd(q, kk, v, alpha, dout, k, per, S, mode)
        got = [np.concatenate([res[r][ci][j] for r in range(2)], axis=2) for j in range(6)]
        for name, a, b in zip(("out", "lse", "dq", "dk", "dv", "dalpha"), got, (out, lse, dq, dk, dv, dal)):
            np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12, err_msg=f"case {ci} {name}")
