"""Ragged (token-pruned) bidirectional attention for ViTs on GB300 (sm_103a).

The compute lives in ``librra.so`` (CUDA kernels behind a C ABI, declared in
``include/rra.h``); ``ragged_attention_token_gb300.rra`` is a thin ctypes
binding with the same names.  Importing this package does not load the
library; the first call into ``rra`` does, and fails loudly if it is missing.
"""
__all__ = ["rra", "workloads"]
