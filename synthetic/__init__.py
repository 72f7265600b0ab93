"""Seeded synthetic inputs shared by the oracle, the tests and the benchmark.

This package only draws random numbers and stores them in the weight formats
the models are defined in (bf16 / fp16 bit patterns, int32 token ids).  It
holds none of the decode arithmetic: no normalisation, attention, rotation,
quantisation or matrix products live here.
"""
from .configs import WORKLOADS, Workload, get_workload  # noqa: F401
from .gen import (  # noqa: F401
    TENSOR_ORDER,
    generate_weights,
    generate_prompt,
    bits_to_f32,
)
