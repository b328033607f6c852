"""Sequence sharding of pi-Attention over devices: the halo plan and its exchange.

The "pi-Attention" page (section 2, item 2) notes that the periodic skips suit strided
gathers or collective communication, and its efficiency results come from 8 GPUs.  With the
sequence split into contiguous shards, one per rank, a shard's queries [t0, t1) attend

    band   [t0 - k, t1)                                   (causal; bidirectional: to t1 + k)
    skips  [t0 - m*period, t1 - m*period) for m = 1..S    with m*period > k (bidirectional:
                                                          also [t0 + m*period, t1 + m*period))
    ECP    [(floor(t0 / c) - 1) * c, t1)                  (the previous half-segment)

clipped to [0, N).  The rows of these sets that another rank owns are the shard's halo.  The
forward receives them point to point (NCCL send/recv on GPUs; gloo, through host copies for device
tensors, in the tests), places them in
a local key/value window [w0, w1) (rows of the window that no query attends stay zero) and runs
pi_attn_fwd_shard on it.  The backward runs pi_attn_bwd_shard, which gives the shard's part of
the window rows' dk/dv, sends the halo rows' parts back to their owners and adds what it
receives to its own rows.  There is no collective beyond these point-to-point transfers.

Everything here is host logic and data movement (torch.distributed, tensor copies); the
attention itself runs in the library's kernels through the binding.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Callable, List, Optional, Tuple

import torch
import torch.distributed as dist

from . import _binding

MODE_PI, MODE_ECP, MODE_PI_BIDIR = _binding.MODE_PI, _binding.MODE_ECP, _binding.MODE_PI_BIDIR
ROW_ALIGN = 128  # shard boundaries and window starts: the kernels' query blocks stay aligned

Interval = Tuple[int, int]


def _merge(iv: List[Interval]) -> List[Interval]:
    out: List[Interval] = []
    for a, b in sorted(x for x in iv if x[1] > x[0]):
        if out and a <= out[-1][1]:
            out[-1] = (out[-1][0], max(out[-1][1], b))
        else:
            out.append((a, b))
    return out


def needed_keys(t0: int, t1: int, N: int, k_local: int, period: int, S: int, mode: int) -> List[Interval]:
    """Key rows the queries [t0, t1) attend, as sorted disjoint half-open intervals of [0, N)."""
    if not 0 <= t0 < t1 <= N:
        raise ValueError(f"bad query range [{t0}, {t1}) for N = {N}")
    clip = lambda a, b: (max(0, a), min(N, b))  # noqa: E731
    if mode == MODE_ECP:
        return _merge([clip((t0 // k_local - 1) * k_local, t1)])
    if mode not in (MODE_PI, MODE_PI_BIDIR):
        raise ValueError(f"unknown mode {mode}")
    hi = t1 + k_local if mode == MODE_PI_BIDIR else t1
    iv = [clip(t0 - k_local, hi)]
    for m in range(1, S + 1):
        off = m * period
        if off <= k_local:
            continue  # inside the band already
        iv.append(clip(t0 - off, t1 - off))
        if mode == MODE_PI_BIDIR:
            iv.append(clip(t0 + off, t1 + off))
    return _merge(iv)


@dataclass(frozen=True)
class Piece:
    """Rows [a, b) (global positions) moving between this rank and `peer`."""
    peer: int
    a: int
    b: int


@dataclass(frozen=True)
class ShardPlan:
    rank: int
    t0: int                      # owned rows [t0, t1): queries and keys/values
    t1: int
    w0: int                      # local key/value window [w0, w1)
    w1: int
    recv: Tuple[Piece, ...] = field(default=())  # halo rows owned by peers (forward: received)
    send: Tuple[Piece, ...] = field(default=())  # own rows in peers' halos (forward: sent)

    @property
    def q_offset(self) -> int:
        return self.t0 - self.w0

    @property
    def n_rows(self) -> int:
        return self.t1 - self.t0

    @property
    def n_window(self) -> int:
        return self.w1 - self.w0


def split(N: int, world: int, align: int = ROW_ALIGN) -> List[Interval]:
    """Contiguous shards of [0, N), one per rank, boundaries on multiples of `align`."""
    if world <= 0 or N <= 0:
        raise ValueError("N and world must be positive")
    units = -(-N // align)  # align-row units, the last one possibly ragged
    if units < world:
        raise ValueError(f"N = {N} is too short for {world} shards of {align}-row multiples")
    base, extra = divmod(units, world)
    bounds, t = [], 0
    for r in range(world):
        n = (base + (r < extra)) * align
        bounds.append((t, min(N, t + n)))
        t += n
    return bounds


def plan(N: int, world: int, k_local: int, period: int, S: int, mode: int,
         align: int = ROW_ALIGN) -> List[ShardPlan]:
    """Every rank's owned rows, window and halo transfers (the same list on every rank)."""
    if mode == MODE_ECP and k_local <= 0:
        raise ValueError("ECP needs the half-segment length c = k_local > 0")
    bounds = split(N, world, align)
    # the window start: a multiple of the row alignment and, in ECP mode, of c, so that the
    # neighbour sets inside the window are those of the whole sequence shifted by w0
    w_align = align if mode != MODE_ECP else align * k_local // math.gcd(align, k_local)
    need = [needed_keys(t0, t1, N, k_local, period, S, mode) for (t0, t1) in bounds]
    recv: List[List[Piece]] = [[] for _ in range(world)]
    send: List[List[Piece]] = [[] for _ in range(world)]
    for r, iv in enumerate(need):
        for (a, b) in iv:
            for src, (s0, s1) in enumerate(bounds):
                lo, hi = max(a, s0), min(b, s1)
                if src == r or lo >= hi:
                    continue
                recv[r].append(Piece(src, lo, hi))
                send[src].append(Piece(r, lo, hi))
    plans = []
    for r, (t0, t1) in enumerate(bounds):
        w0 = min(t0, need[r][0][0]) // w_align * w_align
        w1 = max(t1, need[r][-1][1])
        order = lambda p: (p.a, p.peer)  # noqa: E731  the same order on both ends of a pair
        plans.append(ShardPlan(r, t0, t1, w0, w1, tuple(sorted(recv[r], key=order)),
                               tuple(sorted(send[r], key=order))))
    return plans


# ---------------------------------------------------------------- point-to-point transfers

def _peer(group, r: int) -> int:
    return r if group is None else dist.get_global_rank(group, r)


def _run(ops):
    if ops:
        for w in dist.batch_isend_irecv(ops):
            w.wait()


def _staged(x: torch.Tensor, group) -> bool:
    """Whether transfers of x go through host memory: gloo moves CPU tensors only."""
    return x.is_cuda and dist.get_backend(group) == "gloo"


def _exchange(sends, recvs, dtype, device, group, staged):
    """Point-to-point transfers: sends = [(peer, tensor)], recvs = [(peer, shape)]; returns the
    received tensors on `device`.  With staged, both sides of each transfer are host copies."""
    ops, bufs = [], []
    for peer, t in sends:
        t = t.contiguous()
        ops.append(dist.P2POp(dist.isend, t.cpu() if staged else t, _peer(group, peer), group))
    for peer, shape in recvs:
        buf = torch.empty(shape, dtype=dtype, device="cpu" if staged else device)
        bufs.append(buf)
        ops.append(dist.P2POp(dist.irecv, buf, _peer(group, peer), group))
    _run(ops)
    return [b.to(device) if staged else b for b in bufs]


def gather_window(x_own: torch.Tensor, p: ShardPlan, group=None) -> torch.Tensor:
    """The window [w0, w1) of a [B, Hkv, rows, d] tensor from this rank's rows and the halo
    rows the peers send (rows of the window no query attends are zero)."""
    B, Hkv, n, d = x_own.shape
    if n != p.n_rows:
        raise ValueError(f"rank {p.rank} owns {p.n_rows} rows, got {n}")
    win = torch.zeros((B, Hkv, p.n_window, d), dtype=x_own.dtype, device=x_own.device)
    win[:, :, p.t0 - p.w0:p.t1 - p.w0] = x_own
    got = _exchange([(pc.peer, x_own[:, :, pc.a - p.t0:pc.b - p.t0]) for pc in p.send],
                    [(pc.peer, (B, Hkv, pc.b - pc.a, d)) for pc in p.recv],
                    x_own.dtype, x_own.device, group, _staged(x_own, group))
    for pc, buf in zip(p.recv, got):
        win[:, :, pc.a - p.w0:pc.b - p.w0] = buf
    return win


def reduce_window_grad(g_win: torch.Tensor, p: ShardPlan, group=None) -> torch.Tensor:
    """The reverse of gather_window for gradients: the halo rows' parts go back to their owners,
    and this rank's rows get its own part plus every part received (summed in fp32)."""
    B, Hkv, n, d = g_win.shape
    if n != p.n_window:
        raise ValueError(f"rank {p.rank} has a {p.n_window}-row window, got {n}")
    acc = torch.float64 if g_win.dtype == torch.float64 else torch.float32
    own = g_win[:, :, p.t0 - p.w0:p.t1 - p.w0].to(acc)
    # rows received in the forward send their gradient parts back; rows sent get the peers' parts
    got = _exchange([(pc.peer, g_win[:, :, pc.a - p.w0:pc.b - p.w0]) for pc in p.recv],
                    [(pc.peer, (B, Hkv, pc.b - pc.a, d)) for pc in p.send],
                    g_win.dtype, g_win.device, group, _staged(g_win, group))
    for pc, buf in zip(p.send, got):
        own[:, :, pc.a - p.t0:pc.b - p.t0] += buf.to(acc)
    return own.to(g_win.dtype)


def window_from_full(x_full: torch.Tensor, p: ShardPlan) -> torch.Tensor:
    """The window gather_window builds, taken from a whole-sequence [B, Hkv, N, d] tensor held
    by one process (the rank's own rows and its halo rows; the rest of the window zero)."""
    B, Hkv, _, d = x_full.shape
    win = torch.zeros((B, Hkv, p.n_window, d), dtype=x_full.dtype, device=x_full.device)
    for a, b in [(p.t0, p.t1)] + [(pc.a, pc.b) for pc in p.recv]:
        win[:, :, a - p.w0:b - p.w0] = x_full[:, :, a:b]
    return win


# ---------------------------------------------------------------- forward and backward

@dataclass
class ShardContext:
    plan: ShardPlan
    k_win: torch.Tensor
    v_win: torch.Tensor
    q: torch.Tensor
    alpha: Optional[torch.Tensor]
    out: torch.Tensor
    lse: torch.Tensor
    k_local: int
    period: int
    S: int
    mode: int
    group: object = None


def forward(q, k, v, alpha, p: ShardPlan, k_local: int, period: int, S: int, mode: int = MODE_PI,
            group=None, attend: Optional[Callable] = None):
    """This rank's shard of the forward.  q [B,H,rows,d], k/v [B,Hkv,rows,d], alpha [B,H,rows]:
    the rank's own rows.  Returns (out, lse, ctx) for the rank's rows; ctx feeds backward().
    `attend` has the signature of the binding's fwd_shard, which it defaults to."""
    k_win = gather_window(k, p, group)
    v_win = gather_window(v, p, group)
    fn = attend or _binding.fwd_shard
    out, lse = fn(q, k_win, v_win, alpha, p.q_offset, k_local, period, S, mode)
    return out, lse, ShardContext(p, k_win, v_win, q, alpha, out, lse, k_local, period, S, mode, group)


def backward(ctx: ShardContext, dout, attend_bwd: Optional[Callable] = None):
    """This rank's shard of the backward: (dq, dk, dv, dalpha) of its own rows, dk/dv summed
    over every shard whose queries attend them.  `attend_bwd` defaults to the binding's
    bwd_shard."""
    fn = attend_bwd or _binding.bwd_shard
    dq, dk_win, dv_win, dalpha = fn(ctx.q, ctx.k_win, ctx.v_win, ctx.alpha, ctx.out, ctx.lse, dout,
                                    ctx.plan.q_offset, ctx.k_local, ctx.period, ctx.S, ctx.mode)
    dk = reduce_window_grad(dk_win, ctx.plan, ctx.group)
    dv = reduce_window_grad(dv_win, ctx.plan, ctx.group)
    return dq, dk, dv, dalpha


def halo_rows(p: ShardPlan) -> int:
    """Rows this rank receives in the forward (and sends back in the backward)."""
    return sum(pc.b - pc.a for pc in p.recv)
