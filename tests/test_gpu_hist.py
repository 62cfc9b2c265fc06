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

import oracle
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


def test_histogram_scales_beyond_fp16_fall_back_per_tile():
    """Weights of 32768 on bags that repeat rows: an entry of H (the sum of a
    bag's scales of one row) passes fp16's 65504, so that tile goes to the
    fp32 gather; bags of distinct rows stay on the tensor cores."""
    g = torch.Generator().manual_seed(11)
    tables = [(torch.randn((256, 32), generator=g) * 0.01).half().to(DEV)]
    B = 400
    rng = np.random.default_rng(12)
    lens = rng.integers(1, 40, B)
    idx = []
    for b in range(B):
        if b < 128:  # first tile: rows drawn from 4, so repeats
            idx.append(rng.integers(0, 4, lens[b]))
        else:  # other tiles: distinct rows in each bag
            idx.append(rng.permutation(256)[:lens[b]])
    ind = torch.tensor(np.concatenate(idx), dtype=torch.int64)
    off = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int64)
    w = torch.full((ind.numel(),), 32768.0)  # exact in fp16; two of them are not
    h = tbe.tbe_create(tables, "sum")
    assert tbe.tbe_table_paths(h) == ["histogram"]
    out = tbe.tbe_forward(h, ind.to(DEV), off.to(DEV), B, w.to(DEV))
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    ref, _ = oracle_forward(tables, ind, off, B, w)
    got = out.cpu().numpy()
    # the first tile (fp32 gather) to the fp32 tolerance; the others: exact
    # fp16 H entries and table values, fp32 sums of up to 39 terms of about
    # 330 (rtol 1e-4 and an absolute 1e-2 for outputs that cancel)
    assert_close(got[:128], ref[:128], what="hist overflow tile", **FP32_TOL)
    assert_close(got[128:], ref[128:], what="hist large scales", rtol=1e-4, atol=1e-2)
    h.close()


def test_histogram_bf16_table_beyond_fp16_takes_the_gather():
    """A bf16 table holding values past fp16's range cannot enter the fp16
    MMA: every tile of it is gathered in fp32 (exact to the fp32 tolerance)."""
    g = torch.Generator().manual_seed(13)
    t = torch.randn((128, 16), generator=g) * 0.01
    t[5, 3] = 1.0e6
    tables = [t.bfloat16().to(DEV)]
    B = 200
    ind, off = batch_for(128, B, 30, seed=14)
    h = tbe.tbe_create(tables, "mean")
    assert tbe.tbe_table_paths(h) == ["histogram"]
    out = tbe.tbe_forward(h, ind.to(DEV), off.to(DEV), B)
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    ref, _ = oracle_forward(tables, ind, off, B, None, "mean")
    assert_close(out.cpu().numpy(), ref, what="hist bf16 beyond fp16", **FP32_TOL)
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


# ------------------------------------------------------ dense backward

def _multi_table_batch(specs, B, max_len, seed, oob_table=None):
    """CSR batch over several tables (table-major)."""
    ind, off = [], [torch.zeros(1, dtype=torch.int64)]
    for t, (rows, _, _) in enumerate(specs):
        i, o = batch_for(rows, B, max_len, seed=seed + t, oob=(t == oob_table))
        ind.append(i)
        off.append(o[1:] + off[-1][-1])
    return torch.cat(ind), torch.cat(off)


def _dense_case(specs, B, pooling, weighted, optimizer, flags=0, seed=0, oob_table=None,
                applies=1, max_len=70, index_dtype=torch.int64):
    from helpers import DT_NAME, table_bits, touched_rows, assert_tables_match
    g = torch.Generator().manual_seed(seed)
    tables = [(torch.randn((r, d), generator=g) * 0.01).to(dt).to(DEV) for r, d, dt in specs]
    ind, off = _multi_table_batch(specs, B, max_len, seed=seed + 11, oob_table=oob_table)
    ind, off = ind.to(index_dtype), off.to(index_dtype)
    w = torch.rand(ind.numel(), generator=g) if weighted else None
    grad = torch.randn((B, sum(d for _, d, _ in specs)), generator=g)
    before = [table_bits(t) for t in tables]
    cpu_tables = [t.cpu() for t in tables]
    h = tbe.tbe_create(tables, pooling, flags)
    ws = tbe.make_workspace(h, ind.numel(), B)
    total_rows = sum(r for r, _, _ in specs)
    state = torch.zeros(total_rows, dtype=torch.float32, device=DEV) if optimizer == "adagrad" else None
    tbe.tbe_backward_prepare(h, ind.to(DEV), off.to(DEV), B, ws, None if w is None else w.to(DEV))
    for _ in range(applies):
        tbe.tbe_backward_apply(h, ind.numel(), B, grad.to(DEV), ws, optimizer, 0.05, 1e-8, state)
    rc = tbe.tbe_get_error(h)
    assert rc == (tbe.TBE_ERR_INDEX_OOB if oob_table is not None else tbe.TBE_OK)
    ref_tabs = [table_bits(t) for t in cpu_tables]
    ref_state = None if state is None else np.zeros(total_rows, np.float32)
    for _ in range(applies):
        oracle.backward(ref_tabs, [DT_NAME[t.dtype] for t in cpu_tables], ind.numpy(), off.numpy(), B,
                        grad.numpy(), optimizer, 0.05, eps=1e-8, weights=None if w is None else w.numpy(),
                        pooling=pooling, state=ref_state)
    touched = touched_rows(cpu_tables, ind, off, B)
    assert_tables_match(tables, ref_tabs, before, touched, what=f"dense {specs} {pooling} w={weighted} {optimizer}")
    if state is not None:
        assert_close(state.cpu().numpy(), ref_state, what="dense state", **FP32_TOL)
        st = state.cpu().numpy()
        tm = np.concatenate(touched)
        assert (st[tm] > 0).all() and not st[~tm].any()
    h.close()
    return tables


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("rows,dim", [(512, 64), (100, 16), (33, 48), (300, 128), (512, 256)])
@pytest.mark.parametrize("pooling,weighted", [("sum", False), ("sum", True), ("mean", True)])
def test_dense_backward_sgd_matches_oracle(dtype, rows, dim, pooling, weighted):
    """A histogram table next to a gather-path table: the first takes the
    dense backward, the second the sorted one (compacted keys)."""
    specs = [(rows, dim, dtype), (3000, 32, torch.float32)]
    _dense_case(specs, 333, pooling, weighted, "sgd", seed=rows + dim)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("rows,dim", [(512, 64), (33, 48), (200, 256)])
def test_dense_backward_rowwise_adagrad_matches_oracle(dtype, rows, dim):
    specs = [(700, 64, torch.bfloat16), (rows, dim, dtype), (rows, dim, torch.float16)]
    _dense_case(specs, 257, "mean", True, "adagrad", seed=rows * 3 + dim)


@pytest.mark.parametrize("rows,dim", [(512, 64), (200, 128)])
def test_dense_backward_tiles_past_the_held_lookups(rows, dim):
    """Bags of up to 250 lookups: most 32-bag tiles hold more lookups than the
    per-thread lists cover, so they take the whole-array clears."""
    specs = [(rows, dim, torch.float16), (900, 32, torch.float32)]
    _dense_case(specs, 96, "sum", True, "sgd", seed=rows + 5, max_len=250)


def test_dense_backward_only_dense_tables():
    """Every lookup belongs to a dense table: nothing is sorted."""
    specs = [(512, 64, torch.float16), (128, 32, torch.bfloat16)]
    _dense_case(specs, 300, "sum", True, "adagrad", seed=7)


@pytest.mark.parametrize("index_dtype", [torch.int64, torch.int32])
def test_dense_backward_out_of_range_is_skipped(index_dtype):
    specs = [(64, 32, torch.float16), (5000, 32, torch.float32)]
    _dense_case(specs, 130, "sum", False, "sgd", seed=9, oob_table=0, index_dtype=index_dtype)


def test_dense_backward_applies_twice():
    """prepare once, apply twice: the shared-memory sums start from zero each
    time (the accumulators are cleared per apply).  Each apply is checked as
    one oracle step from the tables it started from (16-bit storage rounds
    after every step, so two oracle steps from the start would compound
    one-ulp differences)."""
    from helpers import DT_NAME, table_bits, touched_rows, assert_tables_match
    specs = [(512, 64, torch.float16), (2000, 64, torch.float32)]
    g = torch.Generator().manual_seed(13)
    tables = [(torch.randn((r, d), generator=g) * 0.01).to(dt).to(DEV) for r, d, dt in specs]
    B = 200
    ind, off = _multi_table_batch(specs, B, 70, seed=24)
    w = torch.rand(ind.numel(), generator=g)
    grad = torch.randn((B, 128), generator=g)
    h = tbe.tbe_create(tables, "sum")
    ws = tbe.make_workspace(h, ind.numel(), B)
    tbe.tbe_backward_prepare(h, ind.to(DEV), off.to(DEV), B, ws, w.to(DEV))
    touched = touched_rows([t.cpu() for t in tables], ind, off, B)
    for step in range(2):
        start = [t.cpu() for t in tables]
        tbe.tbe_backward_apply(h, ind.numel(), B, grad.to(DEV), ws, "sgd", 0.05)
        assert tbe.tbe_get_error(h) == tbe.TBE_OK
        ref = [table_bits(t) for t in start]
        oracle.backward(ref, [DT_NAME[t.dtype] for t in start], ind.numpy(), off.numpy(), B, grad.numpy(), "sgd",
                        0.05, weights=w.numpy())
        assert_tables_match(tables, ref, [table_bits(t) for t in start], touched, what=f"apply {step}")
    h.close()


def test_dense_and_sorted_backward_agree_on_the_histogram_workload():
    """The 65-table workload shrunk: default (dense) and TBE_FLAG_SORTED_BACKWARD
    (sorted) backward both match the oracle."""
    cfg = workloads.get_config(5).scaled(B=300, rows_div=1000, rows_min=512)
    specs = workloads.realize_tables(cfg)
    from helpers import oracle_backward, table_bits, touched_rows, assert_tables_match
    batch = workloads.make_batch(cfg, "cpu", torch.int64, specs)
    grad = workloads.make_grad(cfg, "cpu", specs)
    base = workloads.make_tables(cfg, "cpu", specs)
    ref_tabs, _ = oracle_backward(base, batch.indices, batch.offsets, cfg.B, grad, "sgd", cfg.lr,
                                  weights=batch.weights, pooling=cfg.pooling)
    touched = touched_rows(base, batch.indices, batch.offsets, cfg.B)
    before = [table_bits(t) for t in base]
    for flags in (0, tbe.TBE_FLAG_SORTED_BACKWARD):
        tables = [t.to(DEV) for t in base]
        h = tbe.tbe_create(tables, cfg.pooling, flags)
        ws = tbe.make_workspace(h, batch.N, cfg.B)
        tbe.tbe_backward_sgd(h, batch.indices.to(DEV), batch.offsets.to(DEV), cfg.B, grad.to(DEV), cfg.lr, ws,
                             batch.weights.to(DEV))
        assert tbe.tbe_get_error(h) == tbe.TBE_OK
        assert_tables_match(tables, ref_tabs, before, touched, what=f"workload 5 flags={flags}")
        h.close()
