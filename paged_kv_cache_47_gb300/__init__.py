"""Paged KV-cache decode for GB300 (sm_103a).

The hot path (KV append, split-K paged decode attention with a log-sum-exp
merge, copy-on-write block copy) lives in libpkv, a C-ABI shared library of
hand-written CUDA kernels (include/pkv.h). `binding` is its thin Python
wrapper; `workloads` draws the seeded synthetic decode workloads.
"""
from . import build  # noqa: F401

__all__ = ["build", "binding", "workloads"]
