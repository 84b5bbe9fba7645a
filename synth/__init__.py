"""Seeded synthetic inputs shared by the CUDA path's tests, the oracle's tests and the bench.

This module holds no attention arithmetic: only a counter-based random generator,
the distributions drawn from it, the rounding of fp64 draws to the I/O dtype, and
the workload table (shapes and distributions of the five attention workloads).
"""

from .generate import (  # noqa: F401
    splitmix64,
    uniform01,
    normal,
    to_fp32,
    to_bf16_bits,
    bf16_bits_to_fp32,
    make_qkv,
    Workload,
    WORKLOADS,
    tensor_shapes,
    element_counts,
    make_workload,
)
