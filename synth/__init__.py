"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This package draws random numbers and lays them out; it holds none of the
attention, quantisation or page-scoring arithmetic. Both the CUDA path and the
oracle take their inputs from here, so neither ever feeds the other.
"""
from .workloads import (  # noqa: F401
    WORKLOADS, Workload, SeqData, f32_to_bf16_bits, bf16_bits_to_f32,
    round_to_dtype, make_workload, seq_tokens, queries, block_tables,
    append_tokens, seq_lens, outlier_channels, scaled, cache_kind,
)
