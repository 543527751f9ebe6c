"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This package only draws random inputs in the storage formats the library
consumes; it holds none of the method's arithmetic (no decoding, no GEMM, no
routing, no quantisation of intermediate results).
"""
from .workloads import (  # noqa: F401
    WORKLOADS,
    Workload,
    gen_w4a16,
    gen_fp8_blk128,
    gen_moe,
    generate,
)
