"""GPU: the forward with TBE_FLAG_LENGTH_ORDER (each table's bags pooled in
order of their length) gives bit-identical results to index order, and both
match the oracle: mixed dtypes and row shapes (several bags per warp, one bag
per warp, several column blocks, element-wise rows), empty bags, a bag long
enough for the CTA kernel, a table whose bags are all equally long, weights
and mean pooling, and batch sizes that grow and shrink on one handle."""

import numpy as np
import pytest
import torch

import recommender_sparse_embeddings_gb300 as tbe
from helpers import FP32_TOL, assert_close, oracle_forward

pytestmark = pytest.mark.gpu

DEV = "cuda"

# (rows, dim, dtype): fp16 d64 (four bags a warp), bf16 d128 (two), fp32 d128
# (one), fp32 d512 (two column blocks), bf16 d12 (element-wise)
SPECS = [(700, 64, torch.float16), (900, 128, torch.bfloat16), (800, 128, torch.float32),
         (300, 512, torch.float32), (500, 12, torch.bfloat16)]


def make_tables(seed=0):
    g = torch.Generator().manual_seed(seed)
    return [(torch.randn((r, d), generator=g) * 0.01).to(dt).to(DEV) for r, d, dt in SPECS]


def make_batch(B, seed, long_bag=True, uniform_table=1):
    """Per table, bag lengths uniform in [0, 80] (table `uniform_table`: all
    of length 7); table 0's bag 3 gets 3000 lookups (the CTA kernel)."""
    rng = np.random.default_rng(seed)
    lengths, flat = [], []
    for t, (rows, _, _) in enumerate(SPECS):
        for b in range(B):
            L = 7 if t == uniform_table else int(rng.integers(0, 81))
            if long_bag and t == 0 and b == 3:
                L = 3000
            lengths.append(L)
            flat.extend(rng.integers(0, rows, L).tolist())
    ind = torch.tensor(flat, dtype=torch.int64)
    off = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int64)
    w = torch.rand(len(flat), generator=torch.Generator().manual_seed(seed))
    return ind, off, w


@pytest.mark.parametrize("pooling,weighted", [("sum", False), ("mean", True)])
def test_length_order_bit_identical_and_matches_oracle(pooling, weighted):
    tables = make_tables()
    h_ord = tbe.tbe_create(tables, pooling, tbe.TBE_FLAG_NO_HISTOGRAM | tbe.TBE_FLAG_LENGTH_ORDER)
    h_idx = tbe.tbe_create(tables, pooling, tbe.TBE_FLAG_NO_HISTOGRAM)
    for B, seed in [(1000, 1), (3000, 2), (257, 3), (1000, 4)]:  # grows, shrinks, grows back
        ind, off, w = make_batch(B, seed)
        wd = w.to(DEV) if weighted else None
        got = tbe.tbe_forward(h_ord, ind.to(DEV), off.to(DEV), B, wd)
        base = tbe.tbe_forward(h_idx, ind.to(DEV), off.to(DEV), B, wd)
        assert tbe.tbe_get_error(h_ord) == tbe.TBE_OK
        assert tbe.tbe_get_error(h_idx) == tbe.TBE_OK
        assert torch.equal(got.view(torch.int32), base.view(torch.int32)), f"B={B}: orders differ in bits"
        ref, skipped = oracle_forward(tables, ind, off, B, w if weighted else None, pooling)
        assert skipped == 0
        assert_close(got.cpu().numpy(), ref, what=f"length order B={B}", **FP32_TOL)
    h_ord.close()
    h_idx.close()


def test_length_order_repeated_calls_are_stable():
    """The per-call counters return to zero: the same batch twice gives the
    same bits, after a batch of another shape in between."""
    tables = make_tables(5)
    h = tbe.tbe_create(tables, "sum", tbe.TBE_FLAG_NO_HISTOGRAM | tbe.TBE_FLAG_LENGTH_ORDER)
    ind, off, _ = make_batch(2000, 7)
    first = tbe.tbe_forward(h, ind.to(DEV), off.to(DEV), 2000)
    ind2, off2, _ = make_batch(640, 8, long_bag=False, uniform_table=2)
    tbe.tbe_forward(h, ind2.to(DEV), off2.to(DEV), 640)
    again = tbe.tbe_forward(h, ind.to(DEV), off.to(DEV), 2000)
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    assert torch.equal(first.view(torch.int32), again.view(torch.int32))
    h.close()


@pytest.mark.parametrize("pooling", ["sum", "mean"])
def test_length_order_weight_gradient(pooling):
    """The per-sample weight gradient with the length-keyed order: the same
    bits as index order, and the oracle's values."""
    import oracle
    from helpers import DT_NAME, FP32_TOL, table_bits
    from test_gpu_wgrad import allowance, values
    tables = make_tables(11)
    h_ord = tbe.tbe_create(tables, pooling, tbe.TBE_FLAG_NO_HISTOGRAM | tbe.TBE_FLAG_LENGTH_ORDER)
    h_idx = tbe.tbe_create(tables, pooling, tbe.TBE_FLAG_NO_HISTOGRAM)
    B = 1200
    ind, off, _ = make_batch(B, 12)
    total_d = sum(d for _, d, _ in SPECS)
    grad = torch.randn((B, total_d), generator=torch.Generator().manual_seed(13))
    got = tbe.tbe_per_sample_weight_grad(h_ord, ind.to(DEV), off.to(DEV), B, grad.to(DEV))
    base = tbe.tbe_per_sample_weight_grad(h_idx, ind.to(DEV), off.to(DEV), B, grad.to(DEV))
    assert tbe.tbe_get_error(h_ord) == tbe.TBE_OK
    assert torch.equal(got.view(torch.int32), base.view(torch.int32))
    ref = oracle.weight_grad([table_bits(t) for t in tables], [DT_NAME[t.dtype] for t in tables],
                             ind.numpy(), off.numpy(), B, grad.numpy(), pooling=pooling)
    tol = dict(FP32_TOL)
    tol["atol"] = tol["atol"] + allowance(values(tables), ind.numpy(), off.numpy(), B, grad.numpy(), pooling)
    assert_close(got.cpu().numpy(), ref, what="weight gradient, length order", **tol)
    h_ord.close()
    h_idx.close()
