"""Seeded synthetic inputs for the RMSNorm row workloads.

This package is shared by the fp64 oracle side (tests, CPU baseline) and the
CUDA side (tests, bench). It draws and rounds numbers and nothing else: none
of the normalisation arithmetic lives here.
"""
from .generator import (  # noqa: F401
    WORKLOADS,
    Workload,
    bf16_bits_to_float32,
    float_to_bf16_bits,
    make_inputs,
    storage_to_float64,
    workload,
)
