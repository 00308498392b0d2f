"""Seeded synthetic inputs and random-init head weights.

This package is shared by the CPU oracle's tests and by the GPU path's tests and
benchmark.  It holds no arithmetic of the head itself: it only draws random
numbers, lays out span tables the way the prompt layout of the pages places them,
and rounds float32 draws to bfloat16 storage.
"""
from .bf16 import bf16_to_f32, f32_to_bf16
from .records import Batch, BatchSpec, SparseLexical, make_batch, WORKLOADS, workload_spec
from .weights import HeadShape, make_weights, weight_names

__all__ = [
    "bf16_to_f32", "f32_to_bf16", "Batch", "BatchSpec", "SparseLexical", "make_batch",
    "WORKLOADS", "workload_spec", "HeadShape", "make_weights", "weight_names",
]
