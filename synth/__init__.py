"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This package holds no step of the rolling-KV method: it only draws numbers.
Both the fp64 oracle (through the tests) and the benchmark use it; the CUDA
library carries its own implementation of the same counter-based generator
(``rkv_gen_normal`` in ``include/rkv.h``), which the tests check bit for bit
against this one.
"""
from .generator import (  # noqa: F401
    TAG_Q, TAG_K, TAG_V, TAG_P0, TAG_CLOCK, TAG_PHASE, TAG_FILL,
    splitmix64, counter_key, normal_fp32, normal_bf16_bits, bf16_bits_to_f64,
    f32_to_bf16_bits, token_tensor, uniform_int,
)
from .workloads import WORKLOADS, Workload, workload  # noqa: F401
