"""ctypes binding of libpi_attn.so: argument marshalling only.

Every function here takes torch CUDA tensors, checks that their dtype, layout
and device match what the C ABI expects, and passes raw device pointers, sizes
and the current CUDA stream to the entry point of the same name in
include/pi_attn.h.  Calls only enqueue work; with check=True a compute call also
synchronises its stream and raises if a device-side bounded wait gave up.  All computation runs in the library's CUDA kernels; there
is no fallback: if the library is not built or cannot be loaded, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

MODE_PI = 0
MODE_ECP = 1
MODE_PI_BIDIR = 2  # bidirectional band and skips
PI_OK = 0

_lock = threading.Lock()
_lib = None


class PiAttnError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed: {msg} ({code})")
        self.code = code


def lib_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Load libpi_attn.so (built by structured_sparse_long_gb300.build.build())."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built: {path} is missing; "
                               "run structured_sparse_long_gb300.build.build()")
        lib = ctypes.CDLL(path)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        fwd_args = [P, P, P, P] + [I] * 9 + [P, P, P]
        lib.pi_attn_fwd.argtypes = fwd_args
        lib.pi_attn_fwd_f32.argtypes = fwd_args
        bwd_args = [P, P, P, P, P, P, P] + [I] * 9 + [P, P, P, P, P, Z, P]
        lib.pi_attn_bwd.argtypes = bwd_args
        lib.pi_attn_bwd_f32.argtypes = bwd_args
        lib.pi_attn_bwd_noalloc.argtypes = [P, P, P, P, P, P, P] + [I] * 9 + [P, P, P, P, P]
        lib.pi_attn_bwd_noalloc.restype = I
        lib.pi_attn_bwd_workspace_size.argtypes = [I] * 5
        lib.pi_attn_bwd_workspace_size.restype = Z
        lib.pi_attn_status.argtypes = [P]
        lib.pi_attn_strerror.argtypes = [I]
        lib.pi_attn_strerror.restype = ctypes.c_char_p
        lib.pi_attn_debug_counts.argtypes = [P, P, P, P] + [I] * 10 + [P, P, P, P, P]
        lib.pi_attn_debug_probs.argtypes = [P, P, P, P, P] + [I] * 10 + [P, P, P, P]
        lib.pi_attn_debug_wait_timeout.argtypes = [I, P]
        lib.pi_attn_debug_trace.argtypes = [P, P, P, P] + [I] * 9 + [P, P, P, I, P]
        lib.pi_attn_debug_trace.restype = I
        lib.pi_attn_decode.argtypes = [P, P, P, P] + [I] * 9 + [P, P, P]
        lib.pi_attn_decode.restype = I
        lib.pi_attn_fwd_gated.argtypes = [P, P, P, P, P, P, P] + [I] * 9 + [P, P, P, P]
        lib.pi_attn_fwd_gated.restype = I
        lib.pi_attn_fwd_shard.argtypes = [P, P, P, P] + [I] * 11 + [P, P, P]
        lib.pi_attn_fwd_shard.restype = I
        lib.pi_attn_bwd_shard.argtypes = [P, P, P, P, P, P, P] + [I] * 11 + [P, P, P, P, P, Z, P]
        lib.pi_attn_bwd_shard.restype = I
        for name in ("pi_attn_fwd", "pi_attn_fwd_f32", "pi_attn_bwd", "pi_attn_bwd_f32",
                     "pi_attn_status", "pi_attn_debug_counts", "pi_attn_debug_probs",
                     "pi_attn_debug_wait_timeout"):
            getattr(lib, name).restype = I
        _lib = lib
        return lib


def strerror(code: int) -> str:
    return load().pi_attn_strerror(int(code)).decode()


def _check(fn: str, code: int, stream=None, check: bool = False):
    """Raise on a launch error; with check, also synchronise the stream and raise if a device-side
    bounded wait gave up (the status word, read and cleared by pi_attn_status)."""
    if code != PI_OK:
        raise PiAttnError(fn, code, strerror(code))
    if check:
        st = status(stream)
        if st != PI_OK:
            raise PiAttnError(fn, st, strerror(st))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _expect(t: torch.Tensor, name: str, dtype, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _expect_like(t, name, ref, dtype, shape):
    """A caller-supplied output buffer: a contiguous CUDA tensor of the given dtype and shape on
    the device of `ref` (the kernels store into it with TMA maps sized from the inputs)."""
    _expect(t, name, dtype, shape)
    if t.device != ref.device:
        raise ValueError(f"{name} must be on {ref.device}, got {t.device}")


def _sizes(q, k):
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q must be [B,H,N,d] and k [B,Hkv,N,d]")
    B, H, N, d = q.shape
    return B, H, k.shape[1], N, d


def fwd(q, k, v, alpha, k_local: int, period: int, S: int, mode: int = MODE_PI,
        out=None, lse=None, stream=None, check=False):
    """pi_attn_fwd (bf16) / pi_attn_fwd_f32 (fp32), chosen by q.dtype. Returns (out, lse)."""
    B, H, Hkv, N, d = _sizes(q, k)
    dt = q.dtype
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _expect(t, n, dt)
    _expect(v, "v", dt, k.shape)
    if alpha is not None:
        _expect(alpha, "alpha", torch.float32, (B, H, N))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    _expect(out, "out", dt, q.shape)
    _expect(lse, "lse", torch.float32, (B, H, N))
    lib = load()
    fn = {torch.bfloat16: lib.pi_attn_fwd, torch.float32: lib.pi_attn_fwd_f32}.get(dt)
    if fn is None:
        raise ValueError(f"unsupported dtype {dt}")
    rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), B, H, Hkv, N, d, k_local, period, S, mode,
            _ptr(out), _ptr(lse), _stream(stream))
    _check(fn.__name__, rc, stream, check)
    return out, lse


GATE_HIDDEN = 8  # PI_ATTN_GATE_HIDDEN in include/pi_attn.h


def fwd_gated(q, k, v, gate, k_local: int, period: int, S: int, mode: int = MODE_PI,
              out=None, lse=None, alpha_out=None, stream=None, check=False):
    """pi_attn_fwd_gated (bf16, d 64 or 128): the forward with the gate computed in the same
    launch by the per-head MLP hid = max(0, W1_h q + b1_h), alpha = 1/(1 + exp(-(w2_h . hid + b2_h))).
    gate = (W1 [H, 8, d] bf16, b1 [H, 8], w2 [H, 8], b2 [H] fp32).  Returns (out, lse, alpha)."""
    B, H, Hkv, N, d = _sizes(q, k)
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _expect(t, n, torch.bfloat16)
    _expect(v, "v", torch.bfloat16, k.shape)
    w1, b1, w2, b2 = gate
    _expect(w1, "gate_w1", torch.bfloat16, (H, GATE_HIDDEN, d))
    _expect(b1, "gate_b1", torch.float32, (H, GATE_HIDDEN))
    _expect(w2, "gate_w2", torch.float32, (H, GATE_HIDDEN))
    _expect(b2, "gate_b2", torch.float32, (H,))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    if alpha_out is None:
        alpha_out = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    _expect(out, "out", torch.bfloat16, q.shape)
    _expect(lse, "lse", torch.float32, (B, H, N))
    _expect(alpha_out, "alpha_out", torch.float32, (B, H, N))
    lib = load()
    rc = lib.pi_attn_fwd_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(w1), _ptr(b1), _ptr(w2), _ptr(b2), B, H, Hkv,
                               N, d, k_local, period, S, mode, _ptr(out), _ptr(lse), _ptr(alpha_out),
                               _stream(stream))
    _check("pi_attn_fwd_gated", rc, stream, check)
    return out, lse, alpha_out


def decode(q, k_cache, v_cache, alpha, k_local: int, period: int, S: int, mode: int = MODE_PI,
           out=None, lse=None, stream=None, check=False):
    """pi_attn_decode: q [B,H,d] bf16 against the cache k_cache/v_cache [B,Hkv,N,d] bf16
    (row N-1 of the forward). Returns (out [B,H,d], lse [B,H])."""
    if q.dim() != 3 or k_cache.dim() != 4:
        raise ValueError("q must be [B,H,d] and the caches [B,Hkv,N,d]")
    B, H, d = q.shape
    Hkv, N = k_cache.shape[1], k_cache.shape[2]
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _expect(t, n, torch.bfloat16)
    _expect(v_cache, "v_cache", torch.bfloat16, k_cache.shape)
    if alpha is not None:
        _expect(alpha, "alpha", torch.float32, (B, H))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H), device=q.device, dtype=torch.float32)
    _expect(out, "out", torch.bfloat16, q.shape)
    _expect(lse, "lse", torch.float32, (B, H))
    rc = load().pi_attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(alpha), B, H, Hkv, N, d,
                               k_local, period, S, mode, _ptr(out), _ptr(lse), _stream(stream))
    _check("pi_attn_decode", rc, stream, check)
    return out, lse


def bwd_workspace_size(B, H, Hkv, N, d) -> int:
    return int(load().pi_attn_bwd_workspace_size(B, H, Hkv, N, d))


def _grad_buffers(q, k, v, dq, dk, dv, dalpha):
    """The gradient outputs of the backward: the caller's buffers, checked, or new ones."""
    B, H, N = q.shape[0], q.shape[1], q.shape[2]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if dalpha is None:
        dalpha = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    _expect_like(dq, "dq", q, q.dtype, q.shape)
    _expect_like(dk, "dk", q, q.dtype, k.shape)
    _expect_like(dv, "dv", q, q.dtype, v.shape)
    _expect_like(dalpha, "dalpha", q, torch.float32, (B, H, N))
    return dq, dk, dv, dalpha


def bwd(q, k, v, alpha, out, lse, dout, k_local: int, period: int, S: int, mode: int = MODE_PI,
        dq=None, dk=None, dv=None, dalpha=None, workspace=None, stream=None, check=False):
    """pi_attn_bwd (bf16) / pi_attn_bwd_f32, chosen by q.dtype. Returns (dq, dk, dv, dalpha)."""
    B, H, Hkv, N, d = _sizes(q, k)
    dt = q.dtype
    for t, n in ((q, "q"), (out, "out"), (dout, "dout")):
        _expect(t, n, dt, q.shape)
    for t, n in ((k, "k"), (v, "v")):
        _expect(t, n, dt, k.shape)
    _expect(lse, "lse", torch.float32, (B, H, N))
    if alpha is not None:
        _expect(alpha, "alpha", torch.float32, (B, H, N))
    dq, dk, dv, dalpha = _grad_buffers(q, k, v, dq, dk, dv, dalpha)
    nbytes = bwd_workspace_size(B, H, Hkv, N, d)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), device=q.device, dtype=torch.uint8)
    _expect_like(workspace, "workspace", q, torch.uint8, None)
    if workspace.numel() < nbytes:
        raise ValueError(f"workspace must hold {nbytes} bytes, got {workspace.numel()}")
    lib = load()
    fn = {torch.bfloat16: lib.pi_attn_bwd, torch.float32: lib.pi_attn_bwd_f32}.get(dt)
    if fn is None:
        raise ValueError(f"unsupported dtype {dt}")
    rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(out), _ptr(lse), _ptr(dout),
            B, H, Hkv, N, d, k_local, period, S, mode, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dalpha),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(fn.__name__, rc, stream, check)
    return dq, dk, dv, dalpha


def bwd_noalloc(q, k, v, alpha, out, lse, dout, k_local: int, period: int, S: int,
                mode: int = MODE_PI, dq=None, dk=None, dv=None, dalpha=None, stream=None, check=False):
    """pi_attn_bwd_noalloc (bf16): the backward with the library's fixed device scratch
    instead of a caller workspace.  Returns (dq, dk, dv, dalpha)."""
    B, H, Hkv, N, d = _sizes(q, k)
    for t, n in ((q, "q"), (out, "out"), (dout, "dout")):
        _expect(t, n, torch.bfloat16, q.shape)
    for t, n in ((k, "k"), (v, "v")):
        _expect(t, n, torch.bfloat16, k.shape)
    _expect(lse, "lse", torch.float32, (B, H, N))
    if alpha is not None:
        _expect(alpha, "alpha", torch.float32, (B, H, N))
    dq, dk, dv, dalpha = _grad_buffers(q, k, v, dq, dk, dv, dalpha)
    rc = load().pi_attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(out), _ptr(lse),
                                    _ptr(dout), B, H, Hkv, N, d, k_local, period, S, mode,
                                    _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dalpha), _stream(stream))
    _check("pi_attn_bwd_noalloc", rc, stream, check)
    return dq, dk, dv, dalpha


def _shard_sizes(q, k):
    if q.dim() != 4 or k.dim() != 4 or q.shape[0] != k.shape[0] or q.shape[3] != k.shape[3]:
        raise ValueError("q must be [B,H,Nq,d] and k [B,Hkv,Nkv,d]")
    B, H, Nq, d = q.shape
    return B, H, k.shape[1], Nq, k.shape[2], d


def fwd_shard(q, k, v, alpha, q_offset: int, k_local: int, period: int, S: int, mode: int = MODE_PI,
              out=None, lse=None, stream=None, check=False):
    """pi_attn_fwd_shard (bf16): the queries q [B,H,Nq,d] of a sequence shard, the first at key
    row q_offset of the local key/value window k, v [B,Hkv,Nkv,d].  Returns (out, lse)."""
    B, H, Hkv, Nq, Nkv, d = _shard_sizes(q, k)
    _expect(q, "q", torch.bfloat16)
    _expect(k, "k", torch.bfloat16)
    _expect(v, "v", torch.bfloat16, k.shape)
    if alpha is not None:
        _expect(alpha, "alpha", torch.float32, (B, H, Nq))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), device=q.device, dtype=torch.float32)
    _expect_like(out, "out", q, torch.bfloat16, q.shape)
    _expect_like(lse, "lse", q, torch.float32, (B, H, Nq))
    rc = load().pi_attn_fwd_shard(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), B, H, Hkv, Nq, Nkv,
                                  int(q_offset), d, k_local, period, S, mode, _ptr(out), _ptr(lse),
                                  _stream(stream))
    _check("pi_attn_fwd_shard", rc, stream, check)
    return out, lse


def bwd_shard(q, k, v, alpha, out, lse, dout, q_offset: int, k_local: int, period: int, S: int,
              mode: int = MODE_PI, dq=None, dk=None, dv=None, dalpha=None, workspace=None,
              stream=None, check=False):
    """pi_attn_bwd_shard (bf16).  Returns (dq, dk, dv, dalpha): dq and dalpha of the shard's
    queries, dk and dv [B,Hkv,Nkv,d] the shard's part of the window rows' gradients."""
    B, H, Hkv, Nq, Nkv, d = _shard_sizes(q, k)
    for t, n in ((q, "q"), (out, "out"), (dout, "dout")):
        _expect(t, n, torch.bfloat16, q.shape)
    for t, n in ((k, "k"), (v, "v")):
        _expect(t, n, torch.bfloat16, k.shape)
    _expect(lse, "lse", torch.float32, (B, H, Nq))
    if alpha is not None:
        _expect(alpha, "alpha", torch.float32, (B, H, Nq))
    dq, dk, dv, dalpha = _grad_buffers(q, k, v, dq, dk, dv, dalpha)
    nbytes = bwd_workspace_size(B, H, Hkv, Nq, d)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), device=q.device, dtype=torch.uint8)
    _expect_like(workspace, "workspace", q, torch.uint8, None)
    if workspace.numel() < nbytes:
        raise ValueError(f"workspace must hold {nbytes} bytes, got {workspace.numel()}")
    rc = load().pi_attn_bwd_shard(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(out), _ptr(lse),
                                  _ptr(dout), B, H, Hkv, Nq, Nkv, int(q_offset), d, k_local, period,
                                  S, mode, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dalpha),
                                  _ptr(workspace), workspace.numel(), _stream(stream))
    _check("pi_attn_bwd_shard", rc, stream, check)
    return dq, dk, dv, dalpha


def status(stream=None) -> int:
    """pi_attn_status: synchronise and return (and clear) the device status word."""
    return int(load().pi_attn_status(_stream(stream)))


def debug_counts(q, k, v, alpha, k_local, period, S, mode=MODE_PI, stream=None):
    """pi_attn_debug_counts. Returns (out, lse, count int32 [B,H,N], idx_sum int64 [B,H,N])."""
    B, H, Hkv, N, d = _sizes(q, k)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    cnt = torch.empty((B, H, N), device=q.device, dtype=torch.int32)
    isum = torch.empty((B, H, N), device=q.device, dtype=torch.int64)
    dtype = 1 if q.dtype == torch.float32 else 0
    rc = load().pi_attn_debug_counts(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), B, H, Hkv, N, d,
                                     k_local, period, S, mode, dtype, _ptr(out), _ptr(lse),
                                     _ptr(cnt), _ptr(isum), _stream(stream))
    _check("pi_attn_debug_counts", rc)
    return out, lse, cnt, isum


def debug_probs(q, k, v, alpha, lse_in, k_local, period, S, mode=MODE_PI, stream=None):
    """pi_attn_debug_probs. Returns the dense probabilities P [B,H,N,N] fp32."""
    B, H, Hkv, N, d = _sizes(q, k)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    P = torch.zeros((B, H, N, N), device=q.device, dtype=torch.float32)
    dtype = 1 if q.dtype == torch.float32 else 0
    rc = load().pi_attn_debug_probs(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(lse_in), B, H,
                                    Hkv, N, d, k_local, period, S, mode, dtype, _ptr(out),
                                    _ptr(lse), _ptr(P), _stream(stream))
    _check("pi_attn_debug_probs", rc)
    return P


def debug_trace(q, k, v, alpha, k_local, period, S, mode=MODE_PI, n_ctas=256, stream=None):
    """pi_attn_debug_trace. Returns (out, lse, trace int64 [n_ctas, 240]) of clock64 stamps."""
    B, H, Hkv, N, d = _sizes(q, k)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    trace = torch.zeros((n_ctas, 240), device=q.device, dtype=torch.int64)
    rc = load().pi_attn_debug_trace(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), B, H, Hkv, N, d,
                                    k_local, period, S, mode, _ptr(out), _ptr(lse), _ptr(trace),
                                    n_ctas, _stream(stream))
    _check("pi_attn_debug_trace", rc)
    return out, lse, trace


def debug_wait_timeout(timeout_us: int, stream=None) -> None:
    rc = load().pi_attn_debug_wait_timeout(int(timeout_us), _stream(stream))
    _check("pi_attn_debug_wait_timeout", rc)
