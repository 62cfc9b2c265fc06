"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle on
the same seeded inputs.  Workload shapes follow the five synthetic configs,
shrunk (fewer bags, fewer rows) so the oracle finishes in seconds while the
batches still span many warps, several sort tiles and a ragged tail."""

import types

import numpy as np
import pytest
import torch

import oracle
import recommender_sparse_embeddings_gb300 as tbe
import workloads
from helpers import (FP32_TOL, assert_close, assert_tables_match, oracle_backward, oracle_forward,
                     table_bits, touched_rows, DT_NAME)

pytestmark = pytest.mark.gpu

DEV = "cuda"

# (config id, B, rows divisor, minimum rows)
SCALED = {
    1: (64, 1, 1),
    2: (300, 1000, 64),
    3: (160, 1000, 64),
    4: (256, 1000, 64),
    5: (160, 1000, 512),
}


def scaled_cfg(cid):
    B, div, rmin = SCALED[cid]
    cfg = workloads.get_config(cid)
    return cfg if div == 1 and B == cfg.B else cfg.scaled(B=B, rows_div=div, rows_min=rmin)


def make_problem(cid, index_dtype=torch.int64):
    cfg = scaled_cfg(cid)
    specs = workloads.realize_tables(cfg)
    tables = [t.to(DEV) for t in workloads.make_tables(cfg, "cpu", specs)]
    batch = workloads.make_batch(cfg, "cpu", index_dtype, specs)
    grad = workloads.make_grad(cfg, "cpu", specs)
    return cfg, tables, batch, grad


@pytest.mark.parametrize("index_dtype", [torch.int64, torch.int32])
@pytest.mark.parametrize("cid", [1, 2, 3, 4, 5])
def test_forward_matches_oracle(cid, index_dtype):
    cfg, tables, batch, _ = make_problem(cid, index_dtype)
    h = tbe.tbe_create(tables, cfg.pooling, tbe.TBE_FLAG_NO_HISTOGRAM)
    w = None if batch.weights is None else batch.weights.to(DEV)
    out = tbe.tbe_forward(h, batch.indices.to(DEV), batch.offsets.to(DEV), cfg.B, w)
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    ref, skipped = oracle_forward(tables, batch.indices, batch.offsets, cfg.B, batch.weights, cfg.pooling)
    assert skipped == 0
    assert_close(out.cpu().numpy(), ref, what=f"cfg{cid} forward", **FP32_TOL)


@pytest.mark.parametrize("cid,flags", [(1, 0), (2, 0), (3, 0), (4, 0), (5, 0), (5, tbe.TBE_FLAG_SORTED_BACKWARD)])
def test_prepare_sort_and_rle_bit_exact(cid, flags):
    cfg, tables, batch, _ = make_problem(cid)
    check_prepare(cfg, tables, batch, flags)


@pytest.mark.parametrize("pooling,weighted", [("sum", False), ("sum", True), ("mean", False)])
def test_prepare_compacted_keys_values(pooling, weighted):
    """A small fp16 table takes the dense backward, so only the other two
    tables' keys are sorted (compacted); without per-lookup scales the sort
    carries their flat bags, with weights or mean pooling their positions.
    Bags of 0..50 lookups, a few hot rows for runs past 256."""
    rng = np.random.default_rng(23)
    specs = [(5000, 32, torch.float32), (512, 64, torch.float16), (70000, 64, torch.bfloat16)]
    tables = [torch.zeros((r, d), dtype=dt, device=DEV) for r, d, dt in specs]
    B = 3000
    lens = rng.integers(0, 51, len(specs) * B)
    idx = []
    for t, (r, _, _) in enumerate(specs):
        n = int(lens[t * B:(t + 1) * B].sum())
        ii = rng.integers(0, r, n)
        m = rng.random(n) < 0.1
        ii[m] = rng.integers(0, 4)
        idx.append(ii)
    ind = np.concatenate(idx).astype(np.int64)
    batch = types.SimpleNamespace(
        indices=torch.from_numpy(ind),
        offsets=torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)),
        weights=torch.from_numpy(rng.random(len(ind)).astype(np.float32)) if weighted else None)
    batch.N = len(ind)
    cfg = types.SimpleNamespace(B=B, pooling=pooling)
    h = tbe.tbe_create(tables, pooling)
    assert tbe.tbe_backward_paths(h) == ["sorted", "dense", "sorted"]
    h.close()
    check_prepare(cfg, tables, batch, 0)


def test_prepare_sort_bit_exact_many_waves():
    """A batch of many more 4096-key tiles than one wave of sort CTAs (three
    per SM): the downsweep then ranks by warp match instead of ballots.
    Workload 3's tables (rows / 100) with B = 4096: about 2.5 M lookups,
    20-bit keys, three 8-bit passes."""
    cfg = workloads.get_config(3).scaled(B=4096, rows_div=100, rows_min=64)
    specs = workloads.realize_tables(cfg)
    tables = [t.to(DEV) for t in workloads.make_tables(cfg, "cpu", specs)]
    batch = workloads.make_batch(cfg, "cpu", torch.int64, specs)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert (batch.N + 4095) // 4096 > 3 * sms
    check_prepare(cfg, tables, batch, 0)


def test_prepare_sort_bit_exact_many_waves_9bit_digits():
    """The same beyond one wave with 25-bit keys, which take three 9-bit
    passes: two fp16 tables of 2^24 and 2^20 + 7 rows (dim 16, zeros: the
    preparation reads only the indices), uniform and repeated indices,
    B = 65536 bags of 0..40 lookups."""
    rng = np.random.default_rng(11)
    rows = [1 << 24, (1 << 20) + 7]
    tables = [torch.zeros((r, 16), dtype=torch.float16, device=DEV) for r in rows]
    B = 65536
    lens = rng.integers(0, 41, 2 * B)
    idx = []
    for t, r in enumerate(rows):
        n = int(lens[t * B:(t + 1) * B].sum())
        ii = rng.integers(0, r, n)
        hot = rng.integers(0, r, 8)  # rows repeated often enough for long runs
        m = rng.random(n) < 0.2
        ii[m] = hot[rng.integers(0, 8, int(m.sum()))]
        idx.append(ii)
    batch = types.SimpleNamespace(
        indices=torch.from_numpy(np.concatenate(idx).astype(np.int64)),
        offsets=torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)),
        weights=None)
    batch.N = batch.indices.numel()
    cfg = types.SimpleNamespace(B=B, pooling="sum")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert (batch.N + 4095) // 4096 > 3 * sms
    check_prepare(cfg, tables, batch, 0)


def check_prepare(cfg, tables, batch, flags):
    h = tbe.tbe_create(tables, cfg.pooling, flags)
    ind, off = batch.indices.to(DEV), batch.offsets.to(DEV)
    w = None if batch.weights is None else batch.weights.to(DEV)
    ws = tbe.make_workspace(h, batch.N, cfg.B)
    tbe.tbe_backward_prepare(h, ind, off, cfg.B, ws, w)
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    lay = tbe.tbe_backward_workspace_layout(h, batch.N, cfg.B)
    N = batch.N

    def view(offset, n):
        return ws[offset:offset + 4 * n].view(torch.int32).cpu().numpy().view(np.uint32).astype(np.int64)

    U = int(view(lay.num_unique, 1)[0])
    keys, bag = oracle.make_keys([t.shape[0] for t in tables], batch.indices.numpy(), batch.offsets.numpy(), cfg.B)
    # the small tables' lookups take the dense backward unless
    # TBE_FLAG_SORTED_BACKWARD: only the other tables' keys are sorted (their
    # positions in ascending order)
    dense = np.array([p == "dense" for p in tbe.tbe_backward_paths(h)])
    if flags & tbe.TBE_FLAG_SORTED_BACKWARD:
        assert not dense.any()
    keep = np.flatnonzero(~dense[bag // cfg.B])
    ref = oracle.sort_rle(keys[keep])
    Ns = len(keep)
    np.testing.assert_array_equal(view(lay.sorted_keys, Ns), ref["sorted_keys"])
    # the sorted values: positions when the batch has scales (weights or mean
    # pooling), else the lookups' flat bags
    spos = keep[ref["sorted_pos"]]
    scaled = batch.weights is not None or cfg.pooling == "mean"
    np.testing.assert_array_equal(view(lay.sorted_vals, Ns), spos if scaled else bag[spos])
    assert U == len(ref["uniq"])
    np.testing.assert_array_equal(view(lay.uniq, U), ref["uniq"])
    rs = view(lay.runstart, U + 1)
    np.testing.assert_array_equal(rs[:U], ref["runstart"])
    assert rs[U] == Ns
    np.testing.assert_array_equal(np.diff(rs), ref["runlen"])


@pytest.mark.parametrize("index_dtype,flags", [(torch.int64, 0), (torch.int32, 0),
                                               (torch.int64, tbe.TBE_FLAG_SORTED_BACKWARD)])
@pytest.mark.parametrize("cid", [1, 2, 3, 4, 5])
def test_backward_matches_oracle(cid, index_dtype, flags):
    cfg, tables, batch, grad = make_problem(cid, index_dtype)
    before = [table_bits(t) for t in tables]
    h = tbe.tbe_create(tables, cfg.pooling, flags)
    ind, off = batch.indices.to(DEV), batch.offsets.to(DEV)
    w = None if batch.weights is None else batch.weights.to(DEV)
    ws = tbe.make_workspace(h, batch.N, cfg.B)
    total_rows = sum(t.shape[0] for t in tables)
    state = None
    cpu_tables = [t.cpu() for t in tables]
    if cfg.optimizer == "sgd":
        tbe.tbe_backward_sgd(h, ind, off, cfg.B, grad.to(DEV), cfg.lr, ws, w)
    else:
        state = torch.zeros(total_rows, dtype=torch.float32, device=DEV)
        tbe.tbe_backward_rowwise_adagrad(h, ind, off, cfg.B, grad.to(DEV), state, cfg.lr, cfg.eps, ws, w)
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    ref_tabs, ref_state = oracle_backward(
        cpu_tables, batch.indices, batch.offsets, cfg.B, grad, cfg.optimizer, cfg.lr, cfg.eps,
        batch.weights, cfg.pooling, None if state is None else torch.zeros(total_rows))
    touched = touched_rows(cpu_tables, batch.indices, batch.offsets, cfg.B)
    assert_tables_match(tables, ref_tabs, before, touched, what=f"cfg{cid}")
    if state is not None:
        assert_close(state.cpu().numpy(), ref_state, what=f"cfg{cid} state", **FP32_TOL)
        # one update per row: the state changes exactly at the touched rows
        st = state.cpu().numpy()
        assert (st[np.concatenate(touched)] > 0).all() and not st[~np.concatenate(touched)].any()
