"""Host-only tests of the C ABI: the library builds and loads, exports every
entry point include/pi_attn.h declares, and rejects bad arguments with the
documented status code before launching anything (no GPU needed)."""
import ctypes
import os
import re

import pytest

from structured_sparse_long_gb300 import build as pbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pi_attn.h")

PI_OK, PI_ERR_NULL, PI_ERR_SHAPE, PI_ERR_UNSUPPORTED, PI_ERR_ALIGN, PI_ERR_WORKSPACE = 0, -1, -2, -3, -4, -5


@pytest.fixture(scope="module")
def lib():
    pbuild.build()
    from structured_sparse_long_gb300 import _binding
    return _binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_]+\s*\*?\s*(pi_attn_[a-z0-9_]+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("pi_attn_fwd", "pi_attn_fwd_f32", "pi_attn_bwd", "pi_attn_bwd_f32",
              "pi_attn_bwd_workspace_size", "pi_attn_status", "pi_attn_strerror",
              "pi_attn_debug_counts", "pi_attn_debug_probs", "pi_attn_debug_wait_timeout",
              "pi_attn_decode", "pi_attn_bwd_noalloc", "pi_attn_debug_trace", "pi_attn_fwd_gated",
              "pi_attn_fwd_shard", "pi_attn_bwd_shard"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(pbuild.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), name


def test_strerror(lib):
    assert lib.pi_attn_strerror(0) == b"PI_OK"
    for code in range(-7, 0):
        assert lib.pi_attn_strerror(code).startswith(b"PI_ERR")
    assert b"unknown" in lib.pi_attn_strerror(-99)


def test_workspace_size(lib):
    assert lib.pi_attn_bwd_workspace_size(2, 16, 16, 16384, 64) == 2 * 16 * 16384 * 4
    assert lib.pi_attn_bwd_workspace_size(1, 1, 1, 3, 64) == 256
    assert lib.pi_attn_bwd_workspace_size(0, 1, 1, 3, 64) == 0


A16 = 0x10000  # fake, 16-byte aligned, never dereferenced: validation fails first


def fwd_call(lib, q=A16, k=A16, v=A16, alpha=A16, B=1, H=2, Hkv=2, N=64, d=64, kl=8, per=16, S=1,
             mode=0, out=A16, lse=A16, fn="pi_attn_fwd"):
    return getattr(lib, fn)(q, k, v, alpha, B, H, Hkv, N, d, kl, per, S, mode, out, lse, None)


@pytest.mark.parametrize("fn", ["pi_attn_fwd", "pi_attn_fwd_f32"])
def test_fwd_validation(lib, fn):
    assert fwd_call(lib, q=None, fn=fn) == PI_ERR_NULL
    assert fwd_call(lib, out=None, fn=fn) == PI_ERR_NULL
    assert fwd_call(lib, lse=None, fn=fn) == PI_ERR_NULL
    assert fwd_call(lib, alpha=None, fn=fn) == PI_ERR_NULL          # pi mode needs alpha
    assert fwd_call(lib, B=0, fn=fn) == PI_ERR_SHAPE
    assert fwd_call(lib, N=-1, fn=fn) == PI_ERR_SHAPE
    assert fwd_call(lib, H=3, Hkv=2, fn=fn) == PI_ERR_SHAPE
    assert fwd_call(lib, kl=-1, fn=fn) == PI_ERR_SHAPE
    assert fwd_call(lib, S=-1, fn=fn) == PI_ERR_SHAPE
    assert fwd_call(lib, per=0, S=2, fn=fn) == PI_ERR_SHAPE
    assert fwd_call(lib, mode=1, kl=0, S=0, alpha=None, fn=fn) == PI_ERR_SHAPE   # ECP needs c > 0
    assert fwd_call(lib, mode=1, kl=16, S=1, fn=fn) == PI_ERR_SHAPE               # ECP has no skip
    assert fwd_call(lib, d=48, fn=fn) == PI_ERR_UNSUPPORTED
    assert fwd_call(lib, d=256, fn=fn) == PI_ERR_UNSUPPORTED
    assert fwd_call(lib, mode=3, fn=fn) == PI_ERR_UNSUPPORTED
    assert fwd_call(lib, mode=2, alpha=None, fn=fn) == PI_ERR_NULL   # bidirectional needs alpha
    assert fwd_call(lib, mode=2, per=0, S=2, fn=fn) == PI_ERR_SHAPE
    assert fwd_call(lib, B=1 << 12, H=1 << 10, Hkv=1 << 10, N=1 << 10, fn=fn) == PI_ERR_UNSUPPORTED
    assert fwd_call(lib, q=A16 + 8, fn=fn) == PI_ERR_ALIGN
    assert fwd_call(lib, v=A16 + 2, fn=fn) == PI_ERR_ALIGN
    assert fwd_call(lib, out=A16 + 4, fn=fn) == PI_ERR_ALIGN
    assert fwd_call(lib, lse=A16 + 2, fn=fn) == PI_ERR_ALIGN


def gated_call(lib, q=A16, gw=A16, gb=A16, w2=A16, b2=A16, B=1, H=2, Hkv=2, N=64, d=64, kl=8, per=16,
               S=1, mode=0, out=A16, lse=A16, aout=A16):
    return lib.pi_attn_fwd_gated(q, A16, A16, gw, gb, w2, b2, B, H, Hkv, N, d, kl, per, S, mode, out, lse,
                                 aout, None)


def test_fwd_gated_validation(lib):
    assert gated_call(lib, gw=None) == PI_ERR_NULL
    assert gated_call(lib, gb=None) == PI_ERR_NULL
    assert gated_call(lib, w2=None) == PI_ERR_NULL
    assert gated_call(lib, b2=None) == PI_ERR_NULL
    assert gated_call(lib, w2=A16 + 2) == PI_ERR_ALIGN
    assert gated_call(lib, b2=A16 + 2) == PI_ERR_ALIGN
    assert gated_call(lib, q=None) == PI_ERR_NULL
    assert gated_call(lib, mode=1, kl=16, S=0) == PI_ERR_UNSUPPORTED   # ECP has no gate
    assert gated_call(lib, mode=3) == PI_ERR_UNSUPPORTED
    assert gated_call(lib, d=32) == PI_ERR_UNSUPPORTED                 # tensor-core path only
    assert gated_call(lib, H=3, Hkv=2) == PI_ERR_SHAPE
    assert gated_call(lib, gw=A16 + 4) == PI_ERR_ALIGN                 # float4 loads of w
    assert gated_call(lib, gb=A16 + 2) == PI_ERR_ALIGN
    assert gated_call(lib, aout=A16 + 2) == PI_ERR_ALIGN
    assert gated_call(lib, q=A16 + 8) == PI_ERR_ALIGN


def bwd_call(lib, ws=A16, ws_bytes=1 << 20, dq=A16, alpha=A16, d=64, dalpha=A16, N=64, mode=0,
             fn="pi_attn_bwd"):
    return getattr(lib, fn)(A16, A16, A16, alpha, A16, A16, A16, 1, 2, 2, N, d, 8, 16, 1, mode,
                            dq, A16, A16, dalpha, ws, ws_bytes, None)


@pytest.mark.parametrize("fn", ["pi_attn_bwd", "pi_attn_bwd_f32"])
def test_bwd_validation(lib, fn):
    assert bwd_call(lib, dq=None, fn=fn) == PI_ERR_NULL
    assert bwd_call(lib, alpha=None, fn=fn) == PI_ERR_NULL
    assert bwd_call(lib, d=16, fn=fn) == PI_ERR_UNSUPPORTED
    assert bwd_call(lib, dq=A16 + 8, fn=fn) == PI_ERR_ALIGN
    assert bwd_call(lib, dalpha=A16 + 1, fn=fn) == PI_ERR_ALIGN
    assert bwd_call(lib, ws=None, fn=fn) == PI_ERR_WORKSPACE
    assert bwd_call(lib, ws_bytes=16, fn=fn) == PI_ERR_WORKSPACE
    assert bwd_call(lib, mode=2, alpha=None, fn=fn) == PI_ERR_NULL   # bidirectional needs alpha
    assert bwd_call(lib, mode=2, ws=None, fn=fn) == PI_ERR_WORKSPACE  # validated like pi mode
    assert bwd_call(lib, mode=3, fn=fn) == PI_ERR_UNSUPPORTED


def shard_fwd_call(lib, Nq=128, Nkv=384, off=256, mode=0, kl=8, S=1, q=A16, lse=A16):
    return lib.pi_attn_fwd_shard(q, A16, A16, A16, 1, 2, 2, Nq, Nkv, off, 64, kl, 16, S, mode, A16, lse,
                                 None)


def shard_bwd_call(lib, Nq=128, Nkv=384, off=256, ws_bytes=1 << 20, dq=A16):
    return lib.pi_attn_bwd_shard(A16, A16, A16, A16, A16, A16, A16, 1, 2, 2, Nq, Nkv, off, 64, 8, 16, 1, 0,
                                 dq, A16, A16, A16, A16, ws_bytes, None)


def test_shard_validation(lib):
    """The query window [q_offset, q_offset + Nq) must lie inside the Nkv key rows and start on a
    128-row boundary; the rest is validated as for the whole-sequence calls."""
    assert shard_fwd_call(lib, off=-128) == PI_ERR_SHAPE
    assert shard_fwd_call(lib, off=64) == PI_ERR_SHAPE
    assert shard_fwd_call(lib, off=384) == PI_ERR_SHAPE          # window past the key rows
    assert shard_fwd_call(lib, Nq=0) == PI_ERR_SHAPE
    assert shard_fwd_call(lib, Nq=129) == PI_ERR_SHAPE           # 256 + 129 > 384
    assert shard_fwd_call(lib, Nkv=0) == PI_ERR_SHAPE
    assert shard_fwd_call(lib, q=None) == PI_ERR_NULL
    assert shard_fwd_call(lib, lse=A16 + 2) == PI_ERR_ALIGN
    assert shard_fwd_call(lib, mode=1, kl=16, S=1) == PI_ERR_SHAPE
    assert shard_bwd_call(lib, off=64) == PI_ERR_SHAPE
    assert shard_bwd_call(lib, dq=None) == PI_ERR_NULL
    # the workspace holds one fp32 per query row of the shard (Nq), not per key row
    need = lib.pi_attn_bwd_workspace_size(1, 2, 2, 128, 64)
    assert need < lib.pi_attn_bwd_workspace_size(1, 2, 2, 384, 64)
    assert shard_bwd_call(lib, ws_bytes=need - 1) == PI_ERR_WORKSPACE


def dec_call(lib, q=A16, kc=A16, vc=A16, alpha=A16, B=1, H=4, Hkv=2, N=64, d=64, kl=8, per=16, S=1,
             mode=0, out=A16, lse=A16):
    return lib.pi_attn_decode(q, kc, vc, alpha, B, H, Hkv, N, d, kl, per, S, mode, out, lse, None)


def test_decode_validation(lib):
    assert dec_call(lib, q=None) == PI_ERR_NULL
    assert dec_call(lib, kc=None) == PI_ERR_NULL
    assert dec_call(lib, lse=None) == PI_ERR_NULL
    assert dec_call(lib, alpha=None) == PI_ERR_NULL               # pi mode needs alpha
    assert dec_call(lib, N=0) == PI_ERR_SHAPE
    assert dec_call(lib, H=3, Hkv=2) == PI_ERR_SHAPE
    assert dec_call(lib, mode=1, kl=0, S=0, alpha=None) == PI_ERR_SHAPE
    assert dec_call(lib, mode=2) == PI_ERR_UNSUPPORTED              # bidirectional has no decode
    assert dec_call(lib, d=32) == PI_ERR_UNSUPPORTED
    assert dec_call(lib, H=34, Hkv=2) == PI_ERR_UNSUPPORTED         # 17 query heads per KV head
    assert dec_call(lib, q=A16 + 8) == PI_ERR_ALIGN
    assert dec_call(lib, vc=A16 + 4) == PI_ERR_ALIGN
    assert dec_call(lib, lse=A16 + 2) == PI_ERR_ALIGN


def test_debug_validation(lib):
    assert lib.pi_attn_debug_counts(A16, A16, A16, A16, 1, 2, 2, 64, 64, 8, 16, 1, 0, 0, A16, A16,
                                    None, A16, None) == PI_ERR_NULL
    assert lib.pi_attn_debug_counts(A16, A16, A16, A16, 1, 2, 2, 64, 64, 8, 16, 1, 0, 5, A16, A16,
                                    A16, A16, None) == PI_ERR_UNSUPPORTED
    assert lib.pi_attn_debug_probs(A16, A16, A16, A16, A16, 1, 2, 2, 4096, 64, 8, 16, 1, 0, 0, A16,
                                   A16, A16, None) == PI_ERR_UNSUPPORTED
    assert lib.pi_attn_debug_wait_timeout(0, None) == PI_ERR_SHAPE


def test_binding_fails_loudly_without_cuda():
    """The product path has no CPU fallback: CPU tensors are rejected."""
    import torch
    import structured_sparse_long_gb300 as pa
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    with pytest.raises((ValueError, RuntimeError)):
        pa.fwd(q, q, q, torch.ones(1, 2, 8), 4, 8, 1)
    with pytest.raises((ValueError, RuntimeError)):
        pa.fwd_gated(q, q, q, (torch.zeros(2, 8, 64), torch.zeros(2, 8), torch.zeros(2, 8), torch.zeros(2)), 4, 8, 1)
    with pytest.raises((ValueError, RuntimeError)):
        pa.decode(q[:, :, 0].contiguous(), q, q, torch.ones(1, 2), 4, 8, 1)
    with pytest.raises((ValueError, RuntimeError)):
        pa.bwd(q, q, q, torch.ones(1, 2, 8), q, torch.zeros(1, 2, 8), q, 4, 8, 1)


@pytest.mark.parametrize("bad", ["dq", "dk", "dv", "dalpha"])
@pytest.mark.parametrize("fn", ["bwd", "bwd_noalloc"])
def test_backward_binding_checks_caller_gradient_buffers(monkeypatch, fn, bad):
    """A caller-supplied gradient buffer is checked (device, dtype, shape, layout) before the
    library is reached: the kernels store into it through maps sized from the inputs.  The CUDA
    checks of the inputs are stubbed here (no GPU); the buffer named `bad` is a host tensor or
    has the wrong shape, and the call must stop at it."""
    import torch
    from structured_sparse_long_gb300 import _binding

    real = _binding._expect

    def expect_without_device(t, name, dtype, shape=None):
        if name != bad:
            return
        real(t, name, dtype, shape)  # the bad buffer: a host tensor -> "must be a CUDA tensor"

    monkeypatch.setattr(_binding, "_expect", expect_without_device)
    monkeypatch.setattr(_binding, "load", lambda: pytest.fail("the library was reached"))
    monkeypatch.setattr(_binding, "bwd_workspace_size", lambda *a: 1024)
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    a = torch.ones(1, 2, 8)
    grads = {"dq": q.clone(), "dk": q.clone(), "dv": q.clone(), "dalpha": torch.zeros(1, 2, 8)}
    with pytest.raises(ValueError, match=bad):
        getattr(_binding, fn)(q, q, q, a, q, torch.zeros(1, 2, 8), q, 4, 8, 1, **grads)

    # the same buffer with the wrong shape is refused by the shape check as well
    def expect_shape_only(t, name, dtype, shape=None):
        if name == bad and shape is not None and tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")

    monkeypatch.setattr(_binding, "_expect", expect_shape_only)
    grads[bad] = grads[bad][..., :4].contiguous()  # last dimension cut: wrong shape
    with pytest.raises(ValueError, match=bad):
        getattr(_binding, fn)(q, q, q, a, q, torch.zeros(1, 2, 8), q, 4, 8, 1, **grads)
