"""Seeded generators for TBE inputs, on any torch device.

Everything here is a draw from a seeded torch generator: table values
N(0, init_std) rounded once to the storage dtype, bag lengths from the
per-table law, indices (uniform, or bounded Zipf over a seeded row
permutation), per-sample weights U(0,1), upstream gradients N(0,1).  The CSR
batch layout is table-major: bag (t, b) is flat bag t*B + b and its lookups are
``indices[offsets[t*B+b] : offsets[t*B+b+1]]``.

Draws on "cuda" and on "cpu" use different generator families, so the same
seed gives different values on the two devices; a test that compares two
implementations draws once and hands both the same tensors.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import torch

from .configs import (
    STREAM_GRAD,
    STREAM_INDICES,
    STREAM_LENGTHS,
    STREAM_PERMUTATION,
    STREAM_TABLE_VALUES,
    STREAM_WEIGHTS,
    WorkloadConfig,
    _seed,
    table_specs,
)

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def realize_tables(cfg: WorkloadConfig):
    """The workload's table list (rows, dim, dtype, laws) with its seed applied."""
    return table_specs(cfg)


def _gen(device, cfg_id: int, stream: int, sub: int = 0) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed(cfg_id, stream, sub))
    return g


def zipf_cdf(rows: int, alpha: float, device="cpu") -> torch.Tensor:
    """CDF of the bounded Zipf law p_k ~ k^-alpha over ranks k = 1..rows (float64)."""
    k = torch.arange(1, rows + 1, dtype=torch.float64, device=device)
    w = k.pow(-float(alpha))
    cdf = torch.cumsum(w, 0)
    return cdf / cdf[-1]


def make_tables(cfg: WorkloadConfig, device="cpu", specs=None) -> List[torch.Tensor]:
    """One [rows, dim] tensor per table, N(0, init_std) drawn in fp32 then rounded
    to the storage dtype (round to nearest even)."""
    specs = specs if specs is not None else table_specs(cfg)
    out = []
    for t, s in enumerate(specs):
        g = _gen(device, cfg.cfg_id, STREAM_TABLE_VALUES, t)
        w = torch.randn((s.rows, s.dim), generator=g, device=device, dtype=torch.float32)
        w.mul_(cfg.init_std)
        out.append(w if s.dtype == "f32" else w.to(TORCH_DTYPES[s.dtype]))
        del w
    return out


@dataclass
class Batch:
    indices: torch.Tensor  # [N] int32 | int64
    offsets: torch.Tensor  # [T*B + 1], same dtype as indices
    weights: Optional[torch.Tensor]  # [N] fp32 or None
    lengths: torch.Tensor  # [T*B] int64, bag lengths (offsets differences)
    T: int
    B: int

    @property
    def N(self) -> int:
        return int(self.indices.numel())


def _draw_lengths(spec, B, g, device) -> torch.Tensor:
    kind = spec.length[0]
    if kind == "fixed":
        return torch.full((B,), int(spec.length[1]), dtype=torch.int64, device=device)
    if kind == "poisson":
        mean, lo, hi = spec.length[1], spec.length[2], spec.length[3]
        rate = torch.full((B,), float(mean), dtype=torch.float32, device=device)
        L = torch.poisson(rate, generator=g).to(torch.int64)
        if lo is not None or hi is not None:
            L = L.clamp(min=lo, max=hi)
        return L
    if kind == "uniform":
        lo, hi = int(spec.length[1]), int(spec.length[2])
        return torch.randint(lo, hi + 1, (B,), generator=g, device=device, dtype=torch.int64)
    raise ValueError(f"unknown length law {spec.length!r}")


def _draw_indices(cfg, t, spec, n, device) -> torch.Tensor:
    g = _gen(device, cfg.cfg_id, STREAM_INDICES, t)
    if spec.index[0] == "uniform":
        return torch.randint(0, spec.rows, (n,), generator=g, device=device, dtype=torch.int64)
    if spec.index[0] == "zipf":
        cdf = zipf_cdf(spec.rows, spec.index[1], device=device)
        u = torch.rand((n,), generator=g, device=device, dtype=torch.float64)
        rank = torch.searchsorted(cdf, u, right=True).clamp_(max=spec.rows - 1)
        del cdf, u
        gp = _gen(device, cfg.cfg_id, STREAM_PERMUTATION, t)
        perm = torch.randperm(spec.rows, generator=gp, device=device, dtype=torch.int64)
        return perm[rank]
    raise ValueError(f"unknown index law {spec.index!r}")


def make_batch(cfg: WorkloadConfig, device="cpu", index_dtype=torch.int64,
               specs=None) -> Batch:
    """One CSR batch over all tables (table-major), with optional weights."""
    specs = specs if specs is not None else table_specs(cfg)
    T, B = len(specs), cfg.B
    lengths, idx = [], []
    for t, s in enumerate(specs):
        g = _gen(device, cfg.cfg_id, STREAM_LENGTHS, t)
        L = _draw_lengths(s, B, g, device)
        lengths.append(L)
        idx.append(_draw_indices(cfg, t, s, int(L.sum().item()), device))
    lengths = torch.cat(lengths)
    indices = torch.cat(idx).to(index_dtype)
    del idx
    offsets = torch.zeros(T * B + 1, dtype=torch.int64, device=device)
    torch.cumsum(lengths, 0, out=offsets[1:])
    offsets = offsets.to(index_dtype)
    weights = None
    if cfg.weights:
        gw = _gen(device, cfg.cfg_id, STREAM_WEIGHTS)
        weights = torch.rand((indices.numel(),), generator=gw, device=device,
                             dtype=torch.float32)
    return Batch(indices=indices, offsets=offsets, weights=weights, lengths=lengths, T=T, B=B)


def make_grad(cfg: WorkloadConfig, device="cpu", specs=None) -> torch.Tensor:
    """Upstream gradient of the pooled output, N(0,1) fp32 [B, sum of dims]."""
    specs = specs if specs is not None else table_specs(cfg)
    total_d = sum(s.dim for s in specs)
    g = _gen(device, cfg.cfg_id, STREAM_GRAD)
    return torch.randn((cfg.B, total_d), generator=g, device=device, dtype=torch.float32)
