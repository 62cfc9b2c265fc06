"""The five synthetic TBE workloads, as data.

Each workload fixes the table list (rows, dim, storage dtype), the number of
bags per table B, the per-table bag-length law, the per-table index law, the
pooling mode, whether per-sample weights are present, and the optimizer used
by the backward pass.  Sizes follow the workload descriptions verbatim; the
pages themselves measure on production shard configurations that are not
public, and these seeded inputs stand in for them.

A workload can be shrunk (``scaled``) for parity tests: rows and B shrink, the
laws (Zipf exponent, Poisson mean, one-hot tables, dtype mix) stay the same.
"""

from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np


@dataclass(frozen=True)
class TableSpec:
    """One embedding table and the law its lookups follow.

    length: ("fixed", L) | ("poisson", mean, lo, hi) | ("uniform", lo, hi)
            lo/hi of a Poisson law are an inclusive clip (None = no clip).
    index:  ("uniform",) | ("zipf", alpha)  (Zipf over a seeded row permutation)
    """

    rows: int
    dim: int
    dtype: str  # "f32" | "f16" | "bf16"
    length: tuple
    index: tuple


@dataclass(frozen=True)
class WorkloadConfig:
    cfg_id: int
    name: str
    B: int
    pooling: str  # "sum" | "mean"
    weights: bool
    optimizer: str  # "sgd" | "adagrad"
    lr: float = 0.01
    eps: float = 1e-8
    init_std: float = 0.01
    # Explicit table list, or None when the list itself is drawn from the seed.
    tables: Optional[tuple] = None
    # Parameters of a seed-drawn table list (the mixed-table workload).
    mixed: Optional[dict] = None
    # Shrink factor applied to every table's rows (parity-test variants).
    rows_div: int = 1
    rows_min: int = 1
    description: str = ""
    # the workload prescribes the tensor-core histogram forward for its small
    # tables
    histogram_forward: bool = False

    def scaled(self, B: int, rows_div: int = 1, rows_min: int = 64) -> "WorkloadConfig":
        """Same laws, fewer bags and (optionally) fewer rows per table."""
        return dataclasses.replace(self, B=B, rows_div=rows_div, rows_min=rows_min,
                                   name=f"{self.name}[B={B},rows/{rows_div}]")


def _zipf(alpha):
    return ("zipf", float(alpha))


CONFIGS = {
    1: WorkloadConfig(
        cfg_id=1,
        name="tiny",
        B=64,
        pooling="sum",
        weights=False,
        optimizer="sgd",
        tables=tuple(TableSpec(1000, 16, "f32", ("fixed", 4), ("uniform",)) for _ in range(2)),
        description="T=2 fp32 tables of 1000 rows, dim 16, B=64, pooling factor 4, "
                    "uniform int64 indices, sum pooling, SGD lr=0.01",
    ),
    2: WorkloadConfig(
        cfg_id=2,
        name="t8_fp32_1m_d128_zipf1.05",
        B=8192,
        pooling="sum",
        weights=False,
        optimizer="sgd",
        tables=tuple(TableSpec(1_000_000, 128, "f32", ("poisson", 20.0, 1, 100), _zipf(1.05))
                     for _ in range(8)),
        description="T=8 fp32 tables of 1M rows, dim 128, B=8192, pooling factor "
                    "Poisson(20) clipped to [1,100], Zipf(1.05) indices over a seeded "
                    "row permutation, sum pooling, SGD lr=0.01",
    ),
    3: WorkloadConfig(
        cfg_id=3,
        name="t32_mixed_bf16_fp16_mean_weighted",
        B=16384,
        pooling="mean",
        weights=True,
        optimizer="adagrad",
        mixed=dict(T=32, rows_lo=1e4, rows_hi=1e7, dims=(32, 64, 128, 256),
                   n_bf16=16, n_f16=16, poisson_mean=40.0, alpha=1.1),
        description="T=32 tables, rows log-uniform in [1e4,1e7], dims from "
                    "{32,64,128,256}, 16 bf16 + 16 fp16, B=16384, per-table pooling "
                    "factor 1 (one-hot) or Poisson(40), weights U(0,1), mean pooling, "
                    "Zipf(1.1), row-wise Adagrad lr=0.01 eps=1e-8",
    ),
    4: WorkloadConfig(
        cfg_id=4,
        name="t16_bf16_5m_d128_zipf1.2_hot_rows",
        B=65536,
        pooling="sum",
        weights=False,
        optimizer="adagrad",
        tables=tuple(TableSpec(5_000_000, 128, "bf16", ("fixed", 32), _zipf(1.2))
                     for _ in range(16)),
        description="T=16 bf16 tables of 5M rows, dim 128, B=65536, pooling factor 32, "
                    "Zipf(1.2) indices, sum pooling, row-wise Adagrad",
    ),
    5: WorkloadConfig(
        cfg_id=5,
        name="t64_fp16_512_plus_fp32_20m_histogram",
        B=32768,
        pooling="sum",
        weights=True,
        optimizer="sgd",
        tables=tuple([TableSpec(512, 64, "f16", ("uniform", 1, 64), ("uniform",))
                      for _ in range(64)]
                     + [TableSpec(20_000_000, 128, "f32", ("uniform", 1, 64), ("uniform",))]),
        description="T=64 fp16 tables of 512 rows, dim 64, plus one fp32 table of 20M "
                    "rows, dim 128, B=32768, pooling factor uniform in [1,64], uniform "
                    "indices, weights U(0,1), sum pooling, SGD; the small tables take the "
                    "histogram x table tensor-core forward",
        histogram_forward=True,
    ),
}


def get_config(cfg_id: int) -> WorkloadConfig:
    return CONFIGS[int(cfg_id)]


def _seed(cfg_id: int, stream: int, sub: int = 0) -> int:
    """Deterministic 63-bit seed for (workload, named stream, sub-stream)."""
    state = np.random.SeedSequence([int(cfg_id), int(stream), int(sub)]).generate_state(
        1, dtype=np.uint64)
    return int(state[0]) & ((1 << 63) - 1)


# Named random streams.  Every draw in the generators uses one of these.
STREAM_TABLE_LIST = 1
STREAM_TABLE_VALUES = 2
STREAM_LENGTHS = 3
STREAM_INDICES = 4
STREAM_PERMUTATION = 5
STREAM_WEIGHTS = 6
STREAM_GRAD = 7
STREAM_STATE = 8


def table_specs(cfg: WorkloadConfig) -> list:
    """The realized table list (draws it from the seed for the mixed workload)."""
    if cfg.tables is not None:
        specs = list(cfg.tables)
    else:
        m = cfg.mixed
        rng = np.random.default_rng(_seed(cfg.cfg_id, STREAM_TABLE_LIST))
        T = m["T"]
        log_rows = rng.uniform(math.log(m["rows_lo"]), math.log(m["rows_hi"]), size=T)
        rows = np.rint(np.exp(log_rows)).astype(np.int64)
        dims = rng.choice(np.array(m["dims"]), size=T)
        dtypes = np.array(["bf16"] * m["n_bf16"] + ["f16"] * m["n_f16"])
        rng.shuffle(dtypes)
        onehot = rng.random(T) < 0.5
        specs = []
        for t in range(T):
            length = ("fixed", 1) if onehot[t] else ("poisson", m["poisson_mean"], None, None)
            specs.append(TableSpec(int(rows[t]), int(dims[t]), str(dtypes[t]), length,
                                   _zipf(m["alpha"])))
    if cfg.rows_div != 1:
        specs = [dataclasses.replace(s, rows=max(cfg.rows_min, s.rows // cfg.rows_div))
                 for s in specs]
    return specs
