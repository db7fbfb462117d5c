"""Seeded synthetic inputs shared by the oracle checks, the GPU tests and the bench.

This package only draws random numbers and stores them in the cache's storage
formats. It holds none of the decode step's arithmetic (no bias add, no append,
no attention), so both sides of every parity test can consume it.
"""
from .workloads import (  # noqa: F401
    DTYPE_CODES,
    WORKLOADS,
    Workload,
    gen_all,
    gen_cache_slot,
    gen_qkv,
    gen_scales_slot,
    gen_seq_lens,
    storage_dtype,
    to_storage,
)
