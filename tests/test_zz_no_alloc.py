"""The allocation-free backward entry point, pi_attn_bwd_noalloc.

Some callers cannot give the library a workspace and must not allocate device
memory: a runtime that reserved the device memory up front for its own pool,
code that cannot afford cudaFree's device-wide synchronisation, or bindings
that only forward the buffers they were handed.  For them the backward uses a
fixed device array inside the library instead of a workspace.  These tests call
it through the C ABI and check it against the workspace version, pi_attn_bwd,
on two calls in a row.  The second call runs on different inputs, so that
stale contents of the shared array would show.

This file is collected last on purpose, so that a run that stops at its first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import structured_sparse_long_gb300 as pa
from structured_sparse_long_gb300 import build as pbuild
from structured_sparse_long_gb300.synth import MODE_ECP, MODE_PI, make_inputs, small_case

pytestmark = pytest.mark.gpu

PI_ERR_WORKSPACE = -5
MAX_ROWS = 1 << 20  # PI_ATTN_NOALLOC_MAX_ROWS in include/pi_attn.h
TOL_ABS, TOL_REL = 2e-2, 5e-3  # the bf16 tolerance of the parity tests


@pytest.fixture(scope="module", autouse=True)
def built():
    pbuild.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    pa.load()


def _close(name, a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    max_abs = float(np.abs(a - b).max())
    den = float(np.linalg.norm(b))
    rel = float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a - b))
    assert max_abs <= TOL_ABS and rel <= TOL_REL, f"{name}: max_abs={max_abs:.3e} rel={rel:.3e}"


CASES = [
    small_case("noalloc-a", 1, 4, 2, 300, 64, 40, 64, 2, MODE_PI, "bf16", seed=21, backward=True),
    small_case("noalloc-b", 2, 2, 2, 257, 128, 30, 50, 3, MODE_PI, "bf16", seed=22, backward=True),
    small_case("noalloc-ecp", 1, 2, 1, 200, 64, 48, 0, 0, MODE_ECP, "bf16", seed=23, alpha="none",
               backward=True),
]


def test_noalloc_backward_matches_workspace_backward_on_consecutive_calls():
    for w in CASES:  # consecutive calls share the library's scratch array
        inp = make_inputs(w, with_dout=True)
        d = {n: (t.cuda() if t is not None else None) for n, t in inp.items()}
        out, lse = pa.fwd(d["q"], d["k"], d["v"], d["alpha"], w.k_local, w.period, w.S, w.mode)
        ref = pa.bwd(d["q"], d["k"], d["v"], d["alpha"], out, lse, d["dout"], w.k_local, w.period,
                     w.S, w.mode)
        got = (torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"]),
               torch.empty((w.B, w.H, w.N), device="cuda", dtype=torch.float32))
        pa.bwd_noalloc(d["q"], d["k"], d["v"], d["alpha"], out, lse, d["dout"], w.k_local,
                       w.period, w.S, w.mode, dq=got[0], dk=got[1], dv=got[2], dalpha=got[3])
        torch.cuda.synchronize()
        assert pa.status() == 0
        for name, a, b in zip(("dq", "dk", "dv", "dalpha"), got, ref):
            _close(f"{w.name} {name}", a, b)
            # the same deterministic kernels on the same inputs: identical bits, so that a row
            # of the shared scratch left over from the previous call would show
            assert torch.equal(a, b), f"{w.name} {name}: differs from the workspace backward"


def test_noalloc_rejects_sizes_above_its_scratch():
    """B*H*N above the fixed maximum is refused before anything is touched or launched."""
    lib = pa.load()
    fake = 0x10000  # aligned, never dereferenced: the size check comes first
    B, H, N = 1, 16, MAX_ROWS // 16 + 1
    rc = lib.pi_attn_bwd_noalloc(fake, fake, fake, fake, fake, fake, fake, B, H, H, N, 64, 8, 16, 1,
                                 MODE_PI, fake, fake, fake, fake, None)
    assert rc == PI_ERR_WORKSPACE
    assert pa.strerror(rc).startswith("PI_ERR_WORKSPACE")
    assert isinstance(lib.pi_attn_bwd_noalloc, ctypes._CFuncPtr)
