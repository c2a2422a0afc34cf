"""Seeded synthetic inputs for the QSA sparse-attention step.

This module is shared by the CPU oracle, the tests and the benchmark. It only
draws random numbers and lays them out (cell allocation, block tables, the
q8_0 byte layout of the K/V cache); it holds none of the step's arithmetic
(no pooling, scoring, selection or attention).

Workloads follow the shapes of the llama.cpp qwen4exp issue ("decode slows
linearly with context", fix summary): 16 query heads over 2 KV heads of 256
dims, an indexer with 4 heads of 128 dims, compress_ratio 4, top_k 2048 cells.
"""
from .gen import (  # noqa: F401
    CONFIG_NAMES,
    Step,
    Workload,
    default_cfg,
    make_workload,
    quantize_q8_0,
)
