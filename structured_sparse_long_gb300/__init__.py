"""GB300 (sm_103a) pi-Attention / ECP fused sparse causal attention.

The product is the C-ABI library ``libpi_attn.so`` (include/pi_attn.h) built
from ``csrc/`` for sm_103a.  This package holds that source, the nvcc build
script, a thin ctypes binding with the same names as the C entry points, the
host logic of the sequence-sharded split (``seqshard``: halo plan and point-to-point
exchange), and the seeded synthetic input generators.  Importing the package
loads nothing; the first call loads the library and fails loudly if it is missing.
"""
from ._binding import (MODE_ECP, MODE_PI, MODE_PI_BIDIR, PiAttnError, bwd, bwd_noalloc,  # noqa: F401
                       bwd_shard, bwd_workspace_size, debug_counts, debug_probs, debug_trace,
                       debug_wait_timeout, decode, fwd, fwd_gated, fwd_shard, lib_path, load, status,
                       strerror)

__all__ = ["fwd", "fwd_gated", "fwd_shard", "bwd", "bwd_shard", "decode", "bwd_noalloc",
           "bwd_workspace_size", "status", "strerror", "debug_counts", "debug_probs", "debug_trace",
           "debug_wait_timeout", "load", "lib_path", "PiAttnError", "MODE_PI", "MODE_ECP",
           "MODE_PI_BIDIR"]
