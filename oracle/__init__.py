"""fp64 CPU oracle for pi-Attention / ECP attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The product path (the CUDA library and its Python
binding) never does, and this package never imports the product.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP); this module only
compiles it with gcc, loads it with ctypes and marshals numpy/torch arrays.
Every function follows the plain definition of the method:

* "pi-Attention: Periodic Sparse Transformers for Efficient Long-Context
  Modeling", section 2.1 (ring-local band), 2.2 (pi-skip keys, causal form),
  2.3 (one softmax over the union, gate alpha as log-prior);
* "Efficient Context Propagating Perceiver Architectures for Auto-Regressive
  Language Modeling", section 2 (paired half-segment PAR attention);
* the GQA attention branch of the GSS-Transformer hybrid page (K/V heads
  shared by groups of query heads).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# PI_ORACLE_SRC builds the library from another copy of the C source (into its own directory):
# tests/test_oracle_mutants.py plants one slip in such a copy and checks that the pins fail.
_SRC = os.environ.get("PI_ORACLE_SRC") or os.path.join(_HERE, "oracle.c")
_LIB = (os.path.join(os.path.dirname(os.path.abspath(_SRC)), "liboracle_alt.so")
        if os.environ.get("PI_ORACLE_SRC") else os.path.join(_HERE, "liboracle.so"))
_lock = threading.Lock()
_lib = None

DT_F64, DT_F32, DT_BF16 = 0, 1, 2
MODE_PI, MODE_ECP, MODE_PI_BIDIR = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        L, I, P = ctypes.c_long, ctypes.c_int, ctypes.c_void_p
        lib.oracle_counts.argtypes = [L, I, L, L, I, P, P]
        lib.oracle_counts.restype = None
        lib.oracle_fwd.argtypes = [P, P, P, I, P, L, L, L, L, L, L, L, I, I, L, L, P, P, P]
        lib.oracle_fwd.restype = I
        lib.oracle_bwd.argtypes = [P, P, P, I, P, P, L, L, L, L, L, L, L, I, I, P, P, P, P]
        lib.oracle_bwd.restype = I
        lib.oracle_gate.argtypes = [P, I, P, P, P, P, L, L, L, L, L, P]
        lib.oracle_gate.restype = None
        _lib = lib
        return lib


def _as_raw(t):
    """Return (contiguous numpy array, dtype code) holding the exact input bits."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16), DT_BF16
            if t.dtype == torch.float32:
                return t.numpy(), DT_F32
            if t.dtype == torch.float64:
                return t.numpy(), DT_F64
            raise TypeError(f"unsupported dtype {t.dtype}")
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(t)
    if a.dtype == np.float64:
        return a, DT_F64
    if a.dtype == np.float32:
        return a, DT_F32
    if a.dtype == np.uint16:
        return a, DT_BF16
    raise TypeError(f"unsupported dtype {a.dtype}")


def _alpha(alpha):
    if alpha is None:
        return None
    try:
        import torch
        if isinstance(alpha, torch.Tensor):
            alpha = alpha.detach().cpu().float().contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(alpha, dtype=np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def counts(N, k_local, period, S, mode):
    """Per-row neighbour count and key-index sum (int64 arrays of length N)."""
    lib = _load()
    cnt = np.zeros(N, dtype=np.int64)
    isum = np.zeros(N, dtype=np.int64)
    lib.oracle_counts(N, mode, k_local, period, S, _ptr(cnt), _ptr(isum))
    return cnt, isum


def fwd(q, k, v, alpha, k_local, period, S, mode, rows=None, want_P=False):
    """fp64 forward.  q [B,H,N,d], k/v [B,Hkv,N,d], alpha [B,H,N] or None.

    rows = (i_begin, i_end) restricts the query positions computed (all b, h);
    out then has shape [B,H,i_end-i_begin,d].  want_P returns the dense
    probability tensor [B,H,N,N] as a third value (tiny N only).
    Returns (out, lse[, P]) as float64 numpy arrays.
    """
    lib = _load()
    qa, dt = _as_raw(q)
    ka, dtk = _as_raw(k)
    va, dtv = _as_raw(v)
    assert dt == dtk == dtv, "q, k, v must share a dtype"
    B, H, N, d = qa.shape
    Hkv = ka.shape[1]
    al = _alpha(alpha)
    i0, i1 = (0, N) if rows is None else rows
    out = np.zeros((B, H, i1 - i0, d), dtype=np.float64)
    lse = np.zeros((B, H, i1 - i0), dtype=np.float64)
    P = np.zeros((B, H, N, N), dtype=np.float64) if want_P else None
    rc = lib.oracle_fwd(_ptr(qa), _ptr(ka), _ptr(va), dt, _ptr(al), B, H, Hkv, N, d, k_local,
                        period, S, mode, i0, i1, _ptr(out), _ptr(lse), _ptr(P))
    if rc != 0:
        raise ValueError("oracle_fwd: bad arguments")
    return (out, lse, P) if want_P else (out, lse)


def bwd(q, k, v, alpha, dout, k_local, period, S, mode):
    """fp64 backward.  Returns (dq, dk, dv, dalpha) as float64 numpy arrays."""
    lib = _load()
    qa, dt = _as_raw(q)
    ka, _ = _as_raw(k)
    va, _ = _as_raw(v)
    da, dtd = _as_raw(dout)
    assert dtd == dt, "dout must have the dtype of q"
    B, H, N, d = qa.shape
    Hkv = ka.shape[1]
    al = _alpha(alpha)
    dq = np.zeros((B, H, N, d), dtype=np.float64)
    dk = np.zeros((B, Hkv, N, d), dtype=np.float64)
    dv = np.zeros((B, Hkv, N, d), dtype=np.float64)
    dal = np.zeros((B, H, N), dtype=np.float64)
    rc = lib.oracle_bwd(_ptr(qa), _ptr(ka), _ptr(va), dt, _ptr(al), _ptr(da), B, H, Hkv, N, d,
                        k_local, period, S, mode, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dal))
    if rc != 0:
        raise ValueError("oracle_bwd: bad arguments")
    return dq, dk, dv, dal


def gate(q, w1, b1, w2, b2):
    """Gate alpha [B,H,N] (float64) through the per-head MLP of one hidden layer:
    hid = max(0, W1_h q + b1_h), alpha = 1 / (1 + exp(-(w2_h . hid + b2_h))).

    q [B,H,N,d] (bf16, fp32 or fp64); W1 [H,F,d], b1 [H,F], w2 [H,F], b2 [H] (any float type;
    taken as fp64).  The pi-Attention page, 2.3, names a light network (MLP) per token and per
    head producing alpha from the input content; the head's query is its input here.
    """
    lib = _load()
    qa, dt = _as_raw(q)
    B, H, N, d = qa.shape
    w1a = np.ascontiguousarray(_np64(w1))
    F = w1a.shape[1]
    w1a = w1a.reshape(H, F, d)
    b1a = np.ascontiguousarray(_np64(b1).reshape(H, F))
    w2a = np.ascontiguousarray(_np64(w2).reshape(H, F))
    b2a = np.ascontiguousarray(_np64(b2).reshape(H))
    alpha = np.zeros((B, H, N), dtype=np.float64)
    lib.oracle_gate(_ptr(qa), dt, _ptr(w1a), _ptr(b1a), _ptr(w2a), _ptr(b2a), B, H, N, d, F, _ptr(alpha))
    return alpha


def fwd_gated(q, k, v, gate_weights, k_local, period, S, mode, rows=None):
    """Forward with alpha from the gate (rounded to fp32, the precision the forward takes alpha
    in); gate_weights = (W1, b1, w2, b2).  Returns (out, lse, alpha) with alpha the fp64 gate."""
    alpha = gate(q, *gate_weights)
    out, lse = fwd(q, k, v, alpha.astype(np.float32), k_local, period, S, mode, rows=rows)
    return out, lse, alpha


def _np64(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().cpu().double().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def threads() -> int:
    """OpenMP threads the oracle will use (OMP_NUM_THREADS or all cores)."""
    env = os.environ.get("OMP_NUM_THREADS")
    return int(env) if env else (os.cpu_count() or 1)
