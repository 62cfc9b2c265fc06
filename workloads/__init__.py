"""Seeded synthetic inputs for table-batched embedding (TBE) workloads.

This package only draws inputs: table contents, CSR index batches, per-sample
weights and upstream gradients. It holds none of the operator's arithmetic
(no pooling, no gradient grouping, no optimizer), so that the CPU oracle and
the CUDA path can both consume its output without sharing any computation.
"""

from .configs import CONFIGS, TableSpec, WorkloadConfig, get_config
from .gen import (
    Batch,
    make_batch,
    make_grad,
    make_tables,
    realize_tables,
    zipf_cdf,
)

__all__ = [
    "CONFIGS",
    "TableSpec",
    "WorkloadConfig",
    "get_config",
    "Batch",
    "make_batch",
    "make_grad",
    "make_tables",
    "realize_tables",
    "zipf_cdf",
]
