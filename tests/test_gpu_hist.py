"""GPU parity of the small-table histogram path (tensor cores): the pooled
output of tables the path takes against the CPU oracle.

H holds per-bag sums of lookup scales rounded to the table's 16-bit type
(the tensor cores take both operands in one type), so weighted and mean
pooling carry one 16-bit rounding of each scale; counts (unweighted sum
pooling) stay exact.  The tolerance is the 16-bit one, rtol 1e-2, with an
absolute floor of 1e-4 for tables of N(0, 0.01) values."""

import numpy as np
import pytest
import torch

import recommender_sparse_embeddings_gb300 as tbe
import workloads
from helpers import FP32_TOL, assert_close, oracle_forward

pytestmark = pytest.mark.gpu

DEV = "cuda"
HIST_TOL = dict(rtol=1e-2, atol=1e-4)


def batch_for(rows, B, max_len, seed, oob=False):
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, max_len + 1, B)
    lens[rng.random(B) < 0.1] = 0
    idx = [rng.integers(0, rows, n) for n in lens]
    if oob:
        for ii in idx[::7]:
            if len(ii):
                ii[0] = rows + 5
    ind = torch.tensor(np.concatenate(idx) if idx else np.zeros(0), dtype=torch.int64)
    off = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int64)
    return ind, off


def test_path_selection():
    g = torch.Generator().manual_seed(0)
    mk = lambda r, d, dt: (torch.randn((r, d), generator=g) * 0.01).to(dt).to(DEV)
    tabs = [mk(512, 64, torch.float16), mk(512, 64, torch.bfloat16), mk(512, 64, torch.float32),
            mk(600, 32, torch.float16), mk(100, 24, torch.float16), mk(300, 128, torch.bfloat16)]
    h = tbe.tbe_create(tabs, "sum")
    assert tbe.tbe_table_paths(h) == ["histogram", "histogram", "gather", "gather", "gather", "histogram"]
    h.close()
    h = tbe.tbe_create(tabs, "sum", tbe.TBE_FLAG_FORCE_HISTOGRAM)
    assert tbe.tbe_table_paths(h)[3] == "histogram"
    h.close()
    h = tbe.tbe_create(tabs, "sum", tbe.TBE_FLAG_NO_HISTOGRAM)
    assert "histogram" not in tbe.tbe_table_paths(h)
    h.close()


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("rows,dim", [(512, 64), (100, 16), (33, 48), (300, 128), (512, 32)])
@pytest.mark.parametrize("pooling,weighted", [("sum", False), ("sum", True), ("mean", True)])
def test_histogram_forward_matches_oracle(dtype, rows, dim, pooling, weighted):
    g = torch.Generator().manual_seed(rows * 7 + dim)
    tables = [(torch.randn((rows, dim), generator=g) * 0.01).to(dtype).to(DEV)]
    B = 333  # three tiles of 128 bags, the last one ragged
    ind, off = batch_for(rows, B, 70, seed=rows + dim)
    w = torch.rand(ind.numel(), generator=g) if weighted else None
    h = tbe.tbe_create(tables, pooling)
    assert tbe.tbe_table_paths(h) == ["histogram"]
    out = tbe.tbe_forward(h, ind.to(DEV), off.to(DEV), B, None if w is None else w.to(DEV))
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    ref, _ = oracle_forward(tables, ind, off, B, w, pooling)
    tol = FP32_TOL if (pooling == "sum" and not weighted) else HIST_TOL
    assert_close(out.cpu().numpy(), ref, what=f"hist {dtype} {rows}x{dim} {pooling} w={weighted}", **tol)
    h.close()


def test_histogram_out_of_range_and_int32():
    g = torch.Generator().manual_seed(3)
    tables = [(torch.randn((64, 32), generator=g) * 0.01).half().to(DEV),
              (torch.randn((5000, 32), generator=g) * 0.01).to(DEV)]
    B = 130
    i0, o0 = batch_for(64, B, 40, seed=4, oob=True)
    i1, o1 = batch_for(5000, B, 40, seed=5)
    ind = torch.cat([i0, i1]).to(torch.int32)
    off = torch.cat([o0, o1[1:] + o0[-1]]).to(torch.int32)
    h = tbe.tbe_create(tables, "sum")
    assert tbe.tbe_table_paths(h) == ["histogram", "gather"]
    out = tbe.tbe_forward(h, ind.to(DEV), off.to(DEV), B)
    assert tbe.tbe_get_error(h) == tbe.TBE_ERR_INDEX_OOB
    ref, skipped = oracle_forward(tables, ind, off, B)
    assert skipped > 0
    assert_close(out.cpu().numpy(), ref, what="hist oob", **FP32_TOL)
    h.close()


def test_histogram_workload_small_tables():
    """The 64 fp16 512x64 tables plus one large fp32 table, B shrunk: the small
    tables run on the histogram path, the large one on the gather path."""
    cfg = workloads.get_config(5).scaled(B=300, rows_div=1000, rows_min=512)
    specs = workloads.realize_tables(cfg)
    tables = [t.to(DEV) for t in workloads.make_tables(cfg, "cpu", specs)]
    batch = workloads.make_batch(cfg, "cpu", torch.int64, specs)
    h = tbe.tbe_create(tables, cfg.pooling)
    paths = tbe.tbe_table_paths(h)
    assert paths[:64] == ["histogram"] * 64 and paths[64] == "gather"
    out = tbe.tbe_forward(h, batch.indices.to(DEV), batch.offsets.to(DEV), cfg.B, batch.weights.to(DEV))
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    ref, _ = oracle_forward(tables, batch.indices, batch.offsets, cfg.B, batch.weights, cfg.pooling)
    got = out.cpu().numpy()
    assert_close(got[:, :64 * 64], ref[:, :64 * 64], what="hist tables", **HIST_TOL)
    assert_close(got[:, 64 * 64:], ref[:, 64 * 64:], what="gather table", **FP32_TOL)
    h.close()
