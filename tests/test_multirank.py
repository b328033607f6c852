"""World-size-2 gloo tests (CPU) of the benchmark's multi-rank host logic: the job is
timed by its slowest rank, and the reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        got = bench.reduce_max(10.0 + rank * 5.0, world, "cpu")
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 15.0, 1: 15.0}


def test_reference_arm_silent_off_rank0(capsys):
    import bench

    class A:
        warmup, steps, gpus = 3, 1, 2
    bench.reference_arm(A, bench.WORKLOADS["C1"], rank=1, world=2)
    assert capsys.readouterr().out == ""


def test_work_accounting_matches_closed_forms():
    import bench
    w = bench.WORKLOADS["C4"]
    wk = bench.work(w, False)
    assert wk["pairs"] == 17061760 * 16
    assert wk["fwd_bytes"] == 2 * 268435456 + 2 * 67108864 + 2 * 4 * 16 * 65536
    assert bench.pairs_per_head(8192, 512, 0, 0, 1) == 6033408


def test_work_accounting_of_the_bidirectional_and_gated_workloads():
    """C7 counts the bidirectional pairs (the golden per-head total, from the oracle), forward
    and backward bytes; C8 moves the bytes of C4 (its alpha is written by the gate instead of
    read)."""
    import json
    import os
    import bench
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pair_counts.json")))
    w7 = bench.WORKLOADS["C7"]
    wk7 = bench.work(w7, True)
    assert wk7["pairs"] == gold["workloads"]["C7"]["pairs_per_head"] * w7.B * w7.H
    qo = w7.B * w7.H * w7.N * w7.d * 2
    kv = w7.B * w7.Hkv * w7.N * w7.d * 2
    vec = w7.B * w7.H * w7.N * 4
    assert wk7["bwd_bytes"] == 4 * qo + 4 * kv + 3 * vec
    assert wk7["bwd_flops"] == 8 * w7.d * wk7["pairs"]
    assert bench.work(bench.WORKLOADS["C8"], False) == bench.work(bench.WORKLOADS["C4"], False)


def test_gated_oracle_sample_runs_on_host_cores():
    """The CPU-baseline leg of the gated workload drives the oracle's gate and forward."""
    import bench
    w = bench.WORKLOADS["C8"].replace(N=512)
    smp = bench.OracleSample(w)
    assert smp.run(16) > 0.0


def test_reference_arm_prints_one_contract_line(capsys):
    """Rank 0 of the reference arm (the oracle on host cores) prints one JSON line with the
    contract's keys, its own cpu_baseline and an e2e with no host-device bytes."""
    import json
    import bench

    class A:
        warmup, steps, gpus = 3, 1, 1
    bench.reference_arm(A, bench.WORKLOADS["C1"], rank=0, world=1)
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
                "cpu_baseline", "e2e"):
        assert key in rec, key
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["unit"] == "tokens/s"
    assert rec["config"]["workload"].startswith("C1")
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["value"] == rec["value"]
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["d2h_bytes_per_step"] == 0


def test_kernel_source_hash_ignores_comments_and_layout():
    """Captures stay matched to code, not to comments: the hash's source text drops comments and
    collapses whitespace but keeps string literals (PTX) intact."""
    import bench
    a = 'int x = 1;  // note\n/* block\n comment */ asm("mov.u32 %0, 1; // not a comment");\n'
    b = 'int x = 1;\n\n asm("mov.u32 %0, 1; // not a comment");'
    c = 'int x = 2;\n asm("mov.u32 %0, 1; // not a comment");'
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert "// not a comment" in bench._code_only(a)
