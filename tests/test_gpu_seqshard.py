"""GPU: the shard entry points on one device, each shard with its halo window.

For every shard of a split, the window is built from the whole-sequence tensors exactly as the
halo exchange builds it (own rows and received rows; the rest zero), and pi_attn_fwd_shard /
pi_attn_bwd_shard run on it.  Checks:
  * the shard's out, lse, dq and dalpha equal the whole-sequence call's rows bit for bit (the
    window is aligned so that the kernels walk the same tiles in the same order);
  * out, lse, dq and dalpha match the fp64 oracle of the whole sequence within the bf16
    tolerance of the parity tests;
  * dk and dv, the shards' bf16 window parts summed, differ from the whole-sequence call's by at
    most one bf16 ulp of each part plus one of the whole-sequence value (each bf16 rounding is
    at most half an ulp; the other half covers the fp32 accumulation order), and match the
    oracle in relative L2 error.  Their largest absolute error is not bounded by the parity
    tests' 2e-2: a row held by two shards carries two roundings of parts that can be larger
    than the sum.
"""
import numpy as np
import pytest
import torch

import oracle
import structured_sparse_long_gb300 as pa
from structured_sparse_long_gb300 import build as pbuild
from structured_sparse_long_gb300 import seqshard as ss
from structured_sparse_long_gb300.synth import MODE_ECP, MODE_PI, MODE_PI_BIDIR, make_inputs, small_case

pytestmark = pytest.mark.gpu

TOL_ABS, TOL_REL = 2e-2, 5e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    pbuild.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    pa.load()
    yield
    assert pa.status() == 0


def bf16_ulp(x):
    """Spacing of bfloat16 numbers at |x| (8 significant bits)."""
    return torch.ldexp(torch.ones_like(x, dtype=torch.float32), torch.frexp(x.float()).exponent - 8)


def close(name, got, ref, check_max=True):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{name}: -inf pattern differs"
    diff = np.abs(got[fin] - ref[fin])
    max_abs = float(diff.max()) if diff.size else 0.0
    den = float(np.linalg.norm(ref[fin]))
    rel = float(np.linalg.norm(got[fin] - ref[fin]) / den) if den > 0 else 0.0
    assert (max_abs <= TOL_ABS or not check_max) and rel <= TOL_REL, \
        f"{name}: max_abs={max_abs:.3e} rel={rel:.3e}"


CASES = [  # (case, world)
    (small_case("shard-pi-d64", 1, 4, 2, 1000, 64, 40, 300, 2, MODE_PI, "bf16", seed=61, backward=True), 3),
    (small_case("shard-pi-d128", 1, 8, 2, 1200, 128, 64, 256, 3, MODE_PI, "bf16", seed=62, backward=True), 4),
    (small_case("shard-bidir", 2, 2, 2, 700, 64, 30, 150, 2, MODE_PI_BIDIR, "bf16", seed=63, backward=True), 3),
    (small_case("shard-ecp", 1, 2, 1, 1100, 64, 128, 0, 0, MODE_ECP, "bf16", seed=64, alpha="none",
                backward=True), 3),
    (small_case("shard-d32", 1, 2, 2, 600, 32, 20, 100, 3, MODE_PI, "bf16", seed=65, backward=True), 2),
]


@pytest.mark.parametrize("w,world", CASES, ids=[c[0].name for c in CASES])
def test_shards_with_halo_windows_match_the_whole_sequence(w, world):
    inp = make_inputs(w, with_dout=True)
    d = {n: (t.cuda() if t is not None else None) for n, t in inp.items()}
    full_out, full_lse = pa.fwd(d["q"], d["k"], d["v"], d["alpha"], w.k_local, w.period, w.S, w.mode)
    full = pa.bwd(d["q"], d["k"], d["v"], d["alpha"], full_out, full_lse, d["dout"], w.k_local,
                  w.period, w.S, w.mode)
    dk_sum = torch.zeros(d["k"].shape, device="cuda", dtype=torch.float32)
    dv_sum = torch.zeros_like(dk_sum)
    dk_ulp = bf16_ulp(full[1])
    dv_ulp = bf16_ulp(full[2])
    outs, lses, dqs, dals = [], [], [], []
    for p in ss.plan(w.N, world, w.k_local, w.period, w.S, w.mode):
        rows = slice(p.t0, p.t1)
        q = d["q"][:, :, rows].contiguous()
        al = d["alpha"][:, :, rows].contiguous() if d["alpha"] is not None else None
        k_win = ss.window_from_full(d["k"], p)
        v_win = ss.window_from_full(d["v"], p)
        out, lse = pa.fwd_shard(q, k_win, v_win, al, p.q_offset, w.k_local, w.period, w.S, w.mode)
        dq, dk, dv, dal = pa.bwd_shard(q, k_win, v_win, al, out, lse, d["dout"][:, :, rows].contiguous(),
                                       p.q_offset, w.k_local, w.period, w.S, w.mode)
        torch.cuda.synchronize()
        assert pa.status() == 0
        tag = f"{w.name} shard {p.rank} [{p.t0},{p.t1}) window [{p.w0},{p.w1})"
        assert torch.equal(out, full_out[:, :, rows]), f"{tag}: out differs from the whole sequence"
        assert torch.equal(lse, full_lse[:, :, rows]), f"{tag}: lse differs from the whole sequence"
        assert torch.equal(dq, full[0][:, :, rows]), f"{tag}: dq differs from the whole sequence"
        assert torch.equal(dal, full[3][:, :, rows]), f"{tag}: dalpha differs from the whole sequence"
        dk_sum[:, :, p.w0:p.w1] += dk.float()
        dv_sum[:, :, p.w0:p.w1] += dv.float()
        dk_ulp[:, :, p.w0:p.w1] += bf16_ulp(dk)
        dv_ulp[:, :, p.w0:p.w1] += bf16_ulp(dv)
        outs.append(out)
        lses.append(lse)
        dqs.append(dq)
        dals.append(dal)
    ref_out, ref_lse = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["alpha"], w.k_local, w.period, w.S, w.mode)
    rdq, rdk, rdv, rdal = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["dout"], w.k_local,
                                     w.period, w.S, w.mode)
    cat = lambda ts: torch.cat(ts, dim=2).float().cpu().numpy()  # noqa: E731
    close("out", cat(outs), ref_out)
    close("lse", cat(lses), ref_lse)
    close("dq", cat(dqs), rdq)
    for name, got, whole, ulp, ref in (("dk", dk_sum, full[1], dk_ulp, rdk), ("dv", dv_sum, full[2], dv_ulp, rdv)):
        excess = ((got - whole.float()).abs() - ulp).max().item()
        assert excess <= 0, f"{w.name} {name}: shard sum off the whole-sequence value by {excess:.3e} beyond the bound"
        close(name, got.cpu().numpy(), ref, check_max=False)
    if w.mode != MODE_ECP:
        close("dalpha", cat(dals), rdal)


def test_shard_window_checks():
    """A query window that is not inside the key rows, or not on a 128-row boundary, is refused
    before anything is launched."""
    w = CASES[0][0]
    inp = make_inputs(w, with_dout=False)
    q = inp["q"].cuda()[:, :, :200].contiguous()
    k = inp["k"].cuda()
    v = inp["v"].cuda()
    al = inp["alpha"].cuda()[:, :, :200].contiguous()
    for off in (-128, 64, 900):
        with pytest.raises(pa.PiAttnError) as e:
            pa.fwd_shard(q, k, v, al, off, w.k_local, w.period, w.S, w.mode)
        assert e.value.code == -2  # PI_ERR_SHAPE


# ---------------------------------------------------------------- two ranks through a process group

def _rank(rank, world, port, case_idx, queue):
    import os
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = CASES[case_idx][0]
        inp = make_inputs(w, with_dout=True)
        p = ss.plan(w.N, world, w.k_local, w.period, w.S, w.mode)[rank]
        own = lambda t: None if t is None else t[:, :, p.t0:p.t1].contiguous().cuda()  # noqa: E731
        out, lse, ctx = ss.forward(own(inp["q"]), own(inp["k"]), own(inp["v"]), own(inp["alpha"]), p,
                                   w.k_local, w.period, w.S, w.mode)
        grads = ss.backward(ctx, own(inp["dout"]))
        torch.cuda.synchronize()
        queue.put((rank, pa.status(), [t.cpu() for t in (out, lse) + tuple(grads)]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case_idx", [0, 2])
def test_two_ranks_exchange_halos_through_a_process_group(case_idx):
    """Two ranks (gloo, both on this GPU; their kernels never wait on each other) each hold their
    own rows, exchange halos with seqshard.forward/backward and run the shard kernels.  Their
    results equal, bit for bit, the same plan carried out in one process: out, lse, dq and dalpha
    the whole-sequence rows, dk and dv the owner's window part plus the parts returned to it, in
    the plan's order, summed in fp32."""
    import socket
    import torch.multiprocessing as mp
    w, _ = CASES[case_idx]
    world = 2
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, case_idx, queue)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = {}
    for _ in range(world):
        r, st, ts = queue.get(timeout=600)
        assert st == 0
        res[r] = ts
    for pr in procs:
        pr.join(120)
        assert pr.exitcode == 0

    inp = make_inputs(w, with_dout=True)
    d = {n: (t.cuda() if t is not None else None) for n, t in inp.items()}
    plans = ss.plan(w.N, world, w.k_local, w.period, w.S, w.mode)
    parts = []
    for p in plans:
        rows = slice(p.t0, p.t1)
        q = d["q"][:, :, rows].contiguous()
        al = d["alpha"][:, :, rows].contiguous() if d["alpha"] is not None else None
        kw, vw = ss.window_from_full(d["k"], p), ss.window_from_full(d["v"], p)
        out, lse = pa.fwd_shard(q, kw, vw, al, p.q_offset, w.k_local, w.period, w.S, w.mode)
        dq, dk, dv, dal = pa.bwd_shard(q, kw, vw, al, out, lse, d["dout"][:, :, rows].contiguous(),
                                       p.q_offset, w.k_local, w.period, w.S, w.mode)
        parts.append((out, lse, dq, dk, dv, dal))
    torch.cuda.synchronize()
    assert pa.status() == 0
    for r, p in enumerate(plans):
        got = res[r]
        for j, name in ((0, "out"), (1, "lse"), (2, "dq"), (5, "dalpha")):
            assert torch.equal(got[j], parts[r][j].cpu()), f"rank {r} {name}"
        for j, name in ((3, "dk"), (4, "dv")):
            own = parts[r][j][:, :, p.t0 - p.w0:p.t1 - p.w0].float()
            for pc in p.send:  # the rows of this rank in the peer's window, back from the peer
                q_plan = plans[pc.peer]
                own[:, :, pc.a - p.t0:pc.b - p.t0] += parts[pc.peer][j][:, :, pc.a - q_plan.w0:pc.b - q_plan.w0].float()
            assert torch.equal(got[j], own.to(torch.bfloat16).cpu()), f"rank {r} {name}"
