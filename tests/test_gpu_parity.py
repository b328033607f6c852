"""GPU parity: the CUDA library (through its C ABI) against the fp64 oracle.

Tolerances (stated for this method): bf16 inputs with fp32 accumulation,
max-abs <= 2e-2 and relative L2 <= 5e-3 on out and lse (and on dq, dk, dv,
dalpha for the training workload); fp32 inputs, both <= 1e-5.  Neighbour
enumeration is checked bit-exactly (per-row counts and key-index sums from the
kernels' own tile walk), and the dense probability dump must be exactly zero
outside the union of band and skip keys.
"""
import numpy as np
import pytest
import torch

import oracle
import structured_sparse_long_gb300 as pa
from structured_sparse_long_gb300 import build as pbuild
from structured_sparse_long_gb300.synth import (MODE_ECP, MODE_PI, MODE_PI_BIDIR, WORKLOADS, make_inputs,
                                                small_case)

pytestmark = pytest.mark.gpu

TOL = {"bf16": (2e-2, 5e-3), "f32": (1e-5, 1e-5)}


@pytest.fixture(scope="module", autouse=True)
def built():
    pbuild.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    pa.load()
    yield
    assert pa.status() == 0


def errors(gpu, ref):
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    diff = np.abs(g - r)
    max_abs = float(diff.max()) if diff.size else 0.0
    den = float(np.linalg.norm(r))
    rel = float(np.linalg.norm(g - r) / den) if den > 0 else float(np.linalg.norm(g - r))
    return max_abs, rel


def assert_close(name, gpu, ref, dtype):
    tol_abs, tol_rel = TOL[dtype]
    max_abs, rel = errors(gpu, ref)
    assert max_abs <= tol_abs and rel <= tol_rel, f"{name}: max_abs={max_abs:.3e} rel_l2={rel:.3e}"
    return max_abs, rel


def assert_lse_close(gpu_lse, ref_lse, dtype):
    g = np.asarray(gpu_lse, dtype=np.float64)
    r = np.asarray(ref_lse, dtype=np.float64)
    ninf_r = np.isneginf(r)
    assert np.array_equal(np.isneginf(g), ninf_r), "lse -inf pattern differs"
    assert np.all(np.isfinite(g[~ninf_r])), "non-finite lse"
    return assert_close("lse", g[~ninf_r], r[~ninf_r], dtype)


def run_forward(w, inputs=None):
    inp = inputs or make_inputs(w, with_dout=False)
    dev = {n: (t.cuda() if t is not None else None) for n, t in inp.items()}
    out, lse = pa.fwd(dev["q"], dev["k"], dev["v"], dev["alpha"], w.k_local, w.period, w.S, w.mode)
    torch.cuda.synchronize()
    assert pa.status() == 0
    return inp, dev, out, lse


def check_forward(w, inputs=None):
    inp, dev, out, lse = run_forward(w, inputs)
    ref_out, ref_lse = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["alpha"], w.k_local, w.period,
                                  w.S, w.mode)
    assert_close("out", out.float().cpu().numpy(), ref_out, w.dtype)
    assert_lse_close(lse.cpu().numpy(), ref_lse, w.dtype)
    return inp, dev, out, lse


# ----------------------------------------------------------------------------- the five workloads

@pytest.mark.parametrize("name", ["C1", "C2", "C3", "C4", "C6"])
def test_workload_forward_matches_oracle(name):
    check_forward(WORKLOADS[name])


@pytest.mark.parametrize("name", ["C5", "C7"])
def test_training_forward_and_backward_match_oracle(name):
    """C5 (causal) and C7 (bidirectional): forward, then dq, dk, dv and dalpha, all at full size."""
    w = WORKLOADS[name]
    inp = make_inputs(w, with_dout=True)
    _, dev, out, lse = check_forward(w, inp)
    dq, dk, dv, dal = pa.bwd(dev["q"], dev["k"], dev["v"], dev["alpha"], out, lse, dev["dout"],
                             w.k_local, w.period, w.S, w.mode)
    torch.cuda.synchronize()
    assert pa.status() == 0
    rq, rk, rv, ral = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["dout"], w.k_local,
                                 w.period, w.S, w.mode)
    assert_close("dq", dq.float().cpu().numpy(), rq, "bf16")
    assert_close("dk", dk.float().cpu().numpy(), rk, "bf16")
    assert_close("dv", dv.float().cpu().numpy(), rv, "bf16")
    assert_close("dalpha", dal.cpu().numpy(), ral, "bf16")


# ----------------------------------------------------------------------------- shapes and edges

SMALL = [
    # name, B, H, Hkv, N, d, k, period, S, mode, dtype
    ("ragged-d64", 1, 2, 2, 300, 64, 40, 64, 2, MODE_PI, "bf16"),
    ("ragged-d128", 2, 2, 2, 333, 128, 100, 150, 3, MODE_PI, "bf16"),
    ("gqa4-d128", 1, 8, 2, 257, 128, 64, 96, 4, MODE_PI, "bf16"),
    ("gqa2-d64", 1, 4, 2, 190, 64, 31, 50, 2, MODE_PI, "bf16"),
    ("gqa8-d64", 1, 8, 1, 130, 64, 20, 33, 3, MODE_PI, "bf16"),
    ("gqa3-d64", 1, 6, 2, 150, 64, 17, 40, 2, MODE_PI, "bf16"),
    ("k0", 1, 2, 2, 100, 64, 0, 7, 5, MODE_PI, "bf16"),
    ("S0", 1, 2, 2, 200, 64, 70, 1, 0, MODE_PI, "bf16"),
    ("overlap", 1, 2, 2, 200, 64, 40, 16, 5, MODE_PI, "bf16"),      # m=1,2 inside the band
    ("N<k", 1, 2, 2, 50, 64, 128, 256, 1, MODE_PI, "bf16"),
    ("N<pi", 1, 2, 2, 90, 128, 16, 100, 2, MODE_PI, "bf16"),
    ("tiny-N", 1, 1, 1, 1, 64, 8, 4, 2, MODE_PI, "bf16"),
    ("wide-band", 1, 2, 2, 260, 64, 1000, 8, 2, MODE_PI, "bf16"),
    ("ecp-ragged", 1, 2, 2, 301, 64, 45, 0, 0, MODE_ECP, "bf16"),
    ("ecp-c128-d128", 1, 2, 1, 600, 128, 128, 0, 0, MODE_ECP, "bf16"),
    ("ecp-c1", 1, 2, 2, 70, 64, 1, 0, 0, MODE_ECP, "bf16"),
    ("d32-bf16", 1, 2, 2, 150, 32, 10, 20, 3, MODE_PI, "bf16"),
    ("f32-d64", 1, 2, 1, 200, 64, 30, 40, 2, MODE_PI, "f32"),
    ("f32-d128-ecp", 1, 2, 2, 130, 128, 20, 0, 0, MODE_ECP, "f32"),
    # bidirectional band i-k..i+k and skips i -/+ m*pi
    ("bi-ragged-d64", 1, 2, 2, 300, 64, 40, 64, 2, MODE_PI_BIDIR, "bf16"),
    ("bi-gqa4-d128", 1, 8, 2, 257, 128, 64, 96, 4, MODE_PI_BIDIR, "bf16"),
    ("bi-gqa2-d64", 1, 4, 2, 190, 64, 31, 50, 2, MODE_PI_BIDIR, "bf16"),
    ("bi-k0", 1, 2, 2, 100, 64, 0, 7, 5, MODE_PI_BIDIR, "bf16"),
    ("bi-S0", 1, 2, 2, 200, 64, 70, 1, 0, MODE_PI_BIDIR, "bf16"),
    ("bi-overlap", 1, 2, 2, 200, 64, 40, 16, 5, MODE_PI_BIDIR, "bf16"),
    ("bi-N<k", 1, 2, 2, 50, 64, 128, 256, 1, MODE_PI_BIDIR, "bf16"),
    ("bi-N<pi", 1, 2, 2, 90, 128, 16, 100, 2, MODE_PI_BIDIR, "bf16"),
    ("bi-wide-band", 1, 2, 2, 260, 64, 1000, 8, 2, MODE_PI_BIDIR, "bf16"),
    ("bi-tiny-N", 1, 1, 1, 1, 64, 8, 4, 2, MODE_PI_BIDIR, "bf16"),
    ("bi-long-d128", 1, 4, 1, 1500, 128, 100, 256, 3, MODE_PI_BIDIR, "bf16"),
    ("bi-d32-bf16", 1, 2, 2, 150, 32, 10, 20, 3, MODE_PI_BIDIR, "bf16"),
    ("bi-f32-d64", 1, 2, 1, 200, 64, 30, 40, 2, MODE_PI_BIDIR, "f32"),
]


def small(spec, seed=5, alpha="sigmoid(1.0)"):
    name, B, H, Hkv, N, d, k, per, S, mode, dt = spec
    return small_case(name, B, H, Hkv, N, d, k, per, S, mode, dt, seed=seed,
                      alpha="none" if mode == MODE_ECP else alpha)


@pytest.mark.parametrize("spec", SMALL, ids=[s[0] for s in SMALL])
def test_small_shapes_forward(spec):
    check_forward(small(spec))


@pytest.mark.parametrize("spec", SMALL, ids=[s[0] for s in SMALL])
def test_counts_bit_exact(spec):
    w = small(spec)
    inp = make_inputs(w, with_dout=False)
    dev = {n: (t.cuda() if t is not None else None) for n, t in inp.items()}
    _, _, cnt, isum = pa.debug_counts(dev["q"], dev["k"], dev["v"], dev["alpha"], w.k_local,
                                      w.period, w.S, w.mode)
    torch.cuda.synchronize()
    assert pa.status() == 0
    rc, ri = oracle.counts(w.N, w.k_local, w.period, w.S, w.mode)
    exp_c = np.broadcast_to(rc, (w.B, w.H, w.N))
    exp_i = np.broadcast_to(ri, (w.B, w.H, w.N))
    np.testing.assert_array_equal(cnt.cpu().numpy(), exp_c)
    np.testing.assert_array_equal(isum.cpu().numpy(), exp_i)


@pytest.mark.parametrize("name", ["C1", "C2", "C3", "C4", "C5", "C6", "C7"])
def test_workload_counts_bit_exact(name):
    w = WORKLOADS[name]
    inp = make_inputs(w, with_dout=False)
    dev = {n: (t.cuda() if t is not None else None) for n, t in inp.items()}
    _, _, cnt, isum = pa.debug_counts(dev["q"], dev["k"], dev["v"], dev["alpha"], w.k_local,
                                      w.period, w.S, w.mode)
    torch.cuda.synchronize()
    assert pa.status() == 0
    rc, ri = oracle.counts(w.N, w.k_local, w.period, w.S, w.mode)
    c = cnt.cpu().numpy()
    s = isum.cpu().numpy()
    assert np.array_equal(c, np.broadcast_to(rc, c.shape))
    assert np.array_equal(s, np.broadcast_to(ri, s.shape))


PROB_CASES = [s for s in SMALL if s[4] <= 400 and s[0] in
              ("ragged-d64", "gqa4-d128", "overlap", "ecp-ragged", "d32-bf16", "f32-d64", "N<k",
               "gqa3-d64", "bi-gqa4-d128", "bi-overlap", "bi-f32-d64")]


@pytest.mark.parametrize("spec", PROB_CASES, ids=[s[0] for s in PROB_CASES])
def test_probability_dump(spec):
    w = small(spec)
    inp, dev, out, lse = run_forward(w)
    P = pa.debug_probs(dev["q"], dev["k"], dev["v"], dev["alpha"], lse, w.k_local, w.period, w.S,
                       w.mode)
    torch.cuda.synchronize()
    assert pa.status() == 0
    _, _, Pref = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["alpha"], w.k_local, w.period, w.S,
                            w.mode, want_P=True)
    Pg = P.cpu().numpy()
    assert np.array_equal(Pg == 0.0, Pref == 0.0), "probability support differs from the union"
    tol = 2e-3 if w.dtype == "bf16" else 1e-5
    assert np.abs(Pg - Pref).max() <= tol
    np.testing.assert_allclose(Pg.sum(-1), 1.0, atol=5e-3 if w.dtype == "bf16" else 1e-5)


def test_alpha_edges():
    """alpha = 0 on some rows (band removed; rows without skip keys -> out 0, lse -inf),
    alpha = 1 on others (skip keys removed)."""
    w = small(("edges", 1, 2, 2, 260, 64, 20, 40, 3, MODE_PI, "bf16"))
    inp = make_inputs(w, with_dout=False)
    a = inp["alpha"].clone()
    a[:, 0, ::3] = 0.0
    a[:, 1, ::4] = 1.0
    inp["alpha"] = a
    check_forward(w, inp)
    ff = small(("edges32", 1, 2, 2, 130, 64, 20, 40, 3, MODE_PI, "f32"))
    inp = make_inputs(ff, with_dout=False)
    a = inp["alpha"].clone()
    a[:, 0, ::3] = 0.0
    a[:, 1, ::4] = 1.0
    inp["alpha"] = a
    check_forward(ff, inp)


def test_backward_alpha_edges():
    """The backward where the gate saturates: alpha exactly 0 or 1 on some rows.  One prior is
    then -inf; dalpha there is 0 (a saturated gate passes no gradient), finite everywhere, and
    dq, dk, dv still match the oracle."""
    for spec in (("bedges", 1, 2, 2, 260, 64, 20, 40, 3, MODE_PI, "bf16"),
                 ("bedges128", 1, 4, 2, 200, 128, 30, 50, 2, MODE_PI, "bf16"),
                 ("bedges32", 1, 2, 2, 130, 64, 20, 40, 3, MODE_PI, "f32")):
        w = small(spec).replace(backward=True)
        inp = make_inputs(w, with_dout=True)
        a = inp["alpha"].clone()
        a[:, 0, ::3] = 0.0
        a[:, -1, 1::4] = 1.0
        inp["alpha"] = a
        _, dev, out, lse = run_forward(w, inp)
        dq, dk, dv, dal = pa.bwd(dev["q"], dev["k"], dev["v"], dev["alpha"], out, lse, dev["dout"],
                                 w.k_local, w.period, w.S, w.mode)
        torch.cuda.synchronize()
        assert pa.status() == 0
        dal = dal.cpu()
        assert torch.isfinite(dal).all(), "non-finite dalpha"
        sat = (a == 0.0) | (a == 1.0)
        assert torch.count_nonzero(dal[sat]) == 0, "dalpha must be 0 where the gate saturates"
        rq, rk, rv, ral = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["dout"], w.k_local,
                                     w.period, w.S, w.mode)
        assert np.all(ral[sat.numpy()] == 0.0)
        assert_close(f"{w.name} dq", dq.float().cpu().numpy(), rq, w.dtype)
        assert_close(f"{w.name} dk", dk.float().cpu().numpy(), rk, w.dtype)
        assert_close(f"{w.name} dv", dv.float().cpu().numpy(), rv, w.dtype)
        assert_close(f"{w.name} dalpha", dal.numpy(), ral, w.dtype)


def test_forward_is_deterministic():
    w = WORKLOADS["C2"]
    inp, dev, out1, lse1 = run_forward(w)
    out2, lse2 = pa.fwd(dev["q"], dev["k"], dev["v"], dev["alpha"], w.k_local, w.period, w.S, w.mode)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


BWD_CASES = [
    ("bwd-d64", 1, 2, 2, 200, 64, 30, 48, 3, MODE_PI, "bf16"),
    ("bwd-gqa", 1, 4, 2, 150, 128, 20, 40, 2, MODE_PI, "bf16"),
    ("bwd-ecp", 1, 2, 2, 180, 64, 40, 0, 0, MODE_ECP, "bf16"),
    ("bwd-f32", 1, 2, 1, 120, 64, 16, 24, 3, MODE_PI, "f32"),
    ("bwd-d32", 1, 2, 2, 100, 32, 10, 15, 2, MODE_PI, "bf16"),
    # bidirectional: band i-k..i+k, skips i -/+ m*pi (queries before and after each key)
    ("bwd-bi-d64", 1, 2, 2, 300, 64, 40, 64, 2, MODE_PI_BIDIR, "bf16"),
    ("bwd-bi-gqa-d128", 1, 8, 2, 257, 128, 64, 96, 3, MODE_PI_BIDIR, "bf16"),
    ("bwd-bi-gqa2-d64", 1, 4, 2, 190, 64, 31, 50, 2, MODE_PI_BIDIR, "bf16"),
    ("bwd-bi-k0", 1, 2, 2, 100, 64, 0, 7, 5, MODE_PI_BIDIR, "bf16"),
    ("bwd-bi-S0", 1, 2, 2, 200, 64, 70, 1, 0, MODE_PI_BIDIR, "bf16"),
    ("bwd-bi-overlap", 1, 2, 2, 200, 64, 40, 16, 5, MODE_PI_BIDIR, "bf16"),
    ("bwd-bi-N<pi", 1, 2, 2, 90, 128, 16, 100, 2, MODE_PI_BIDIR, "bf16"),
    ("bwd-bi-long-d128", 1, 4, 1, 1500, 128, 100, 256, 3, MODE_PI_BIDIR, "bf16"),
    ("bwd-bi-f32", 1, 2, 1, 120, 64, 16, 24, 3, MODE_PI_BIDIR, "f32"),
    ("bwd-bi-d32", 1, 2, 2, 100, 32, 10, 15, 2, MODE_PI_BIDIR, "bf16"),
    # blocks whose number of skip multiples grows along the sequence (1 to 6; bidirectional:
    # backward and forward multiples), in one launch
    ("bwd-mixed-skip", 1, 2, 2, 700, 64, 20, 64, 6, MODE_PI, "bf16"),
    ("bwd-bi-mixed-d128", 1, 4, 4, 600, 128, 30, 100, 3, MODE_PI_BIDIR, "bf16"),
    # four query heads per KV head with one skip multiple; 1/sqrt(d) inputs keep dv (a sum over
    # 4 heads) below 8, where bf16 storage alone stays inside the max-abs bound
    ("bwd-gqa4-S1", 1, 8, 2, 300, 128, 40, 64, 1, MODE_PI, "bf16", "inv_sqrt_d"),
]


@pytest.mark.parametrize("spec", BWD_CASES, ids=[s[0] for s in BWD_CASES])
def test_small_backward(spec):
    name, B, H, Hkv, N, d, k, per, S, mode, dt = spec[:11]
    scale = spec[11] if len(spec) > 11 else "unit"
    # fp32 cases draw alpha as the fp32 workload C1 does, U(0.2, 0.8): dalpha carries the factor
    # 1/(alpha (1 - alpha)), and the fp32 bound is absolute
    a_spec = "none" if mode == MODE_ECP else ("uniform(0.2,0.8)" if dt == "f32" else "sigmoid(1.0)")
    w = small_case(name, B, H, Hkv, N, d, k, per, S, mode, dt, seed=9, qkv_scale=scale, alpha=a_spec,
                   backward=True)
    inp = make_inputs(w, with_dout=True)
    dev = {n: (t.cuda() if t is not None else None) for n, t in inp.items()}
    out, lse = pa.fwd(dev["q"], dev["k"], dev["v"], dev["alpha"], k, per, S, mode)
    dq, dk, dv, dal = pa.bwd(dev["q"], dev["k"], dev["v"], dev["alpha"], out, lse, dev["dout"], k,
                             per, S, mode)
    torch.cuda.synchronize()
    assert pa.status() == 0
    rq, rk, rv, ral = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["dout"], k, per, S,
                                 mode)
    assert_close("dq", dq.float().cpu().numpy(), rq, dt)
    assert_close("dk", dk.float().cpu().numpy(), rk, dt)
    assert_close("dv", dv.float().cpu().numpy(), rv, dt)
    has_skip = mode != MODE_ECP and any(k < m * per < N for m in range(1, S + 1))
    if mode != MODE_ECP and not has_skip:
        # No skip key anywhere (S = 0, or every m*pi is inside the band or past N): dalpha is
        # exactly zero, because every softmax row of dz sums to zero.  The oracle's direct chain rule reaches it only up to fp64 rounding, so a
        # relative error would divide by rounding noise; compare the exact zero instead.
        assert np.all(dal.cpu().numpy() == 0.0)
        assert float(np.abs(ral).max()) <= 1e-10
    else:
        assert_close("dalpha", dal.cpu().numpy(), ral, dt)


def test_backward_dq_precision_d128_gqa():
    """A d=128 GQA case (seed 1) whose dq lost accuracy when the bf16 operand of the dq
    accumulation carried p*dp and D*sum(p k) was subtracted afterwards; centring the operand
    on dout.out keeps dq within the bf16 bound."""
    w = small_case("bwd-dq-d128", 1, 8, 2, 300, 128, 64, 96, 3, MODE_PI, "bf16", seed=1,
                   backward=True)
    inp = make_inputs(w, with_dout=True)
    dev = {n: (t.cuda() if t is not None else None) for n, t in inp.items()}
    out, lse = pa.fwd(dev["q"], dev["k"], dev["v"], dev["alpha"], w.k_local, w.period, w.S, w.mode)
    dq, dk, dv, dal = pa.bwd(dev["q"], dev["k"], dev["v"], dev["alpha"], out, lse, dev["dout"],
                             w.k_local, w.period, w.S, w.mode)
    torch.cuda.synchronize()
    assert pa.status() == 0
    rq, rk, rv, ral = oracle.bwd(inp["q"], inp["k"], inp["v"], inp["alpha"], inp["dout"], w.k_local,
                                 w.period, w.S, w.mode)
    assert_close("dq", dq.float().cpu().numpy(), rq, "bf16")
    assert_close("dk", dk.float().cpu().numpy(), rk, "bf16")
    assert_close("dv", dv.float().cpu().numpy(), rv, "bf16")


def test_bounded_wait_reports_timeout_and_context_survives():
    pa.debug_wait_timeout(2000)  # 2 ms on a barrier nothing completes
    assert pa.status() == -7
    assert pa.status() == 0  # reading clears it
    check_forward(WORKLOADS["C1"])  # the context is still usable


def test_checked_call_raises_on_a_device_timeout():
    """check=True: the call synchronises and raises PI_ERR_DEVICE_TIMEOUT when the status word
    holds a bounded wait that gave up (here the probe's); the next checked call is clean."""
    w = small_case("chk", 1, 2, 2, 200, 64, 16, 32, 2, MODE_PI, "bf16", seed=5)
    inp = make_inputs(w, with_dout=False)
    d = {n: (t.cuda() if t is not None else None) for n, t in inp.items()}
    pa.debug_wait_timeout(2000)
    with pytest.raises(pa.PiAttnError) as e:
        pa.fwd(d["q"], d["k"], d["v"], d["alpha"], w.k_local, w.period, w.S, w.mode, check=True)
    assert e.value.code == -7
    out, lse = pa.fwd(d["q"], d["k"], d["v"], d["alpha"], w.k_local, w.period, w.S, w.mode, check=True)
    ref_out, ref_lse = oracle.fwd(inp["q"], inp["k"], inp["v"], inp["alpha"], w.k_local, w.period, w.S,
                                  w.mode)
    assert_close("out", out.float().cpu().numpy(), ref_out, "bf16")


def test_trace_mode_matches_forward_and_stamps_are_ordered():
    """pi_attn_debug_trace runs the same forward: identical out/lse, and per-tile stamps of
    the softmax warp (one clock) are in order."""
    w = WORKLOADS["C2"]
    inp, dev, out, lse = run_forward(w)
    out2, lse2, tr = pa.debug_trace(dev["q"], dev["k"], dev["v"], dev["alpha"], w.k_local, w.period,
                                    w.S, w.mode, n_ctas=64)
    torch.cuda.synchronize()
    assert pa.status() == 0
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    T = tr.cpu().numpy()
    for c in range(64):
        nt = int(T[c, 7])
        assert 1 <= nt <= 16
        for t in range(nt):
            seen, loaded, maxed, stored, ready = (T[c, 72 + t], T[c, 184 + t], T[c, 200 + t],
                                                  T[c, 216 + t], T[c, 88 + t])
            assert 0 < seen <= loaded <= maxed <= stored <= ready
            assert T[c, 168 + t] >= 0 and T[c, 104 + t] >= 0
