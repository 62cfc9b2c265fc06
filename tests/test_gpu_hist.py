"""GPU parity of the small-table histogram path (tensor cores): the pooled
output of tables the path takes against the CPU oracle.

Each histogram entry is summed in fp32 and reaches the tensor cores as two
fp16 terms (scaled per bag into fp16's range; bf16 tables are scaled per
table), so the outputs are held to the fp32 tolerance of the gather path,
rtol 1e-5 and atol 1e-6, plus histogram_allowance: the two-term rounding of
an entry (2^-21 of the output's absolute term sum) and the rounding of an
fp32 sum of L terms.  That allowance only matters where an output cancels
to far below its terms."""

import numpy as np
import pytest
import torch

import oracle
import recommender_sparse_embeddings_gb300 as tbe
import workloads
from helpers import FP32_TOL, assert_close, histogram_allowance, oracle_forward, pooled_abs_sum

pytestmark = pytest.mark.gpu

DEV = "cuda"


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


def check_hist(out, tables, ind, off, B, w=None, pooling="sum", what="", cols=None):
    """Pooled output against the oracle: the fp32 tolerance plus the
    histogram path's allowance (columns `cols` only, when given)."""
    ref, _ = oracle_forward(tables, ind, off, B, w, pooling)
    abs_sum, n = pooled_abs_sum(tables, ind, off, B, w, pooling)
    got = out.cpu().numpy() if isinstance(out, torch.Tensor) else out
    if cols is not None:
        got, ref, abs_sum, n = got[:, cols], ref[:, cols], abs_sum[:, cols], n[:, cols]
    assert_close(got, ref, what=what, rtol=FP32_TOL["rtol"],
                 atol=FP32_TOL["atol"] + histogram_allowance(abs_sum, n))
    return ref


def run_hist(tables, ind, off, B, w=None, pooling="sum", flags=tbe.TBE_FLAG_FORCE_HISTOGRAM, expect=tbe.TBE_OK):
    h = tbe.tbe_create(tables, pooling, flags)
    paths = tbe.tbe_table_paths(h)
    out = tbe.tbe_forward(h, ind.to(DEV), off.to(DEV), B, None if w is None else w.to(DEV))
    assert tbe.tbe_get_error(h) == expect
    h.close()
    return out, paths


def test_path_selection():
    g = torch.Generator().manual_seed(0)
    mk = lambda r, d, dt: (torch.randn((r, d), generator=g) * 0.01).to(dt).to(DEV)
    tabs = [mk(512, 64, torch.float16), mk(512, 64, torch.bfloat16), mk(512, 64, torch.float32),
            mk(600, 32, torch.float16), mk(100, 24, torch.float16), mk(300, 128, torch.bfloat16)]
    # default: every forward on the gather; the small tables' backward dense
    h = tbe.tbe_create(tabs, "sum")
    assert tbe.tbe_table_paths(h) == ["gather"] * 6
    assert tbe.tbe_backward_paths(h) == ["dense", "dense", "sorted", "sorted", "sorted", "dense"]
    h.close()
    h = tbe.tbe_create(tabs, "sum", tbe.TBE_FLAG_SORTED_BACKWARD)
    assert tbe.tbe_backward_paths(h) == ["sorted"] * 6
    h.close()
    # the histogram forward on request; tables of up to 1024 rows are then
    # small.  The tables of one dtype share one launch, so together they must
    # fit one CTA's shared memory (A for the most rows, the largest W^T): the
    # 600-row fp16 table does not fit beside the 512 x 64 one (gather
    # forward, dense backward), alone it does
    h = tbe.tbe_create(tabs, "sum", tbe.TBE_FLAG_FORCE_HISTOGRAM)
    assert tbe.tbe_table_paths(h) == ["histogram", "histogram", "gather", "gather", "gather", "histogram"]
    assert tbe.tbe_backward_paths(h) == ["dense", "dense", "sorted", "dense", "sorted", "dense"]
    h.close()
    h = tbe.tbe_create([tabs[3], tabs[2]], "sum", tbe.TBE_FLAG_FORCE_HISTOGRAM)
    assert tbe.tbe_table_paths(h) == ["histogram", "gather"]
    h.close()
    h = tbe.tbe_create(tabs, "sum", tbe.TBE_FLAG_NO_HISTOGRAM)
    assert "histogram" not in tbe.tbe_table_paths(h)
    assert tbe.tbe_backward_paths(h) == ["sorted"] * 6
    h.close()


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("rows,dim", [(512, 64), (100, 16), (33, 48), (300, 128), (512, 32)])
@pytest.mark.parametrize("pooling,weighted", [("sum", False), ("sum", True), ("mean", True), ("mean", False)])
def test_histogram_forward_matches_oracle(dtype, rows, dim, pooling, weighted):
    g = torch.Generator().manual_seed(rows * 7 + dim)
    tables = [(torch.randn((rows, dim), generator=g) * 0.01).to(dtype).to(DEV)]
    B = 333  # six tiles of 64 bags, the last one ragged
    ind, off = batch_for(rows, B, 70, seed=rows + dim)
    w = torch.rand(ind.numel(), generator=g) if weighted else None
    out, paths = run_hist(tables, ind, off, B, w, pooling)
    assert paths == ["histogram"]
    check_hist(out, tables, ind, off, B, w, pooling, what=f"hist {dtype} {rows}x{dim} {pooling} w={weighted}")


def test_histogram_repeated_row_in_one_bag():
    """Bags of 64 lookups of one row with U(0,1) weights: each H entry is a
    sum of 64 scales (two 32-lookup chunks, each grouped in lane order, then
    added into the entry); the output is that sum times the row."""
    g = torch.Generator().manual_seed(21)
    tables = [(torch.randn((512, 64), generator=g) * 0.01).half().to(DEV)]
    B = 200
    rng = np.random.default_rng(22)
    rows = rng.integers(0, 512, B)
    ind = torch.tensor(np.repeat(rows, 64), dtype=torch.int64)
    off = torch.arange(0, 64 * B + 1, 64, dtype=torch.int64)
    w = torch.rand(ind.numel(), generator=g)
    for pooling in ("sum", "mean"):
        out, paths = run_hist(tables, ind, off, B, w, pooling)
        assert paths == ["histogram"]
        check_hist(out, tables, ind, off, B, w, pooling, what=f"repeated row {pooling}")


def test_histogram_repeated_row_with_cancelling_rows():
    """One row repeated 40 times per bag beside rows of the opposite sign
    (negated copies of it, weighted so the bag's output nearly cancels): the
    output is small against its terms."""
    g = torch.Generator().manual_seed(23)
    base = torch.randn((256, 32), generator=g) * 0.01
    base[128:] = -base[:128]  # row r + 128 is -row r
    tables = [base.half().to(DEV)]
    B = 150
    rng = np.random.default_rng(24)
    idx, wts = [], []
    for b in range(B):
        r = int(rng.integers(0, 128))
        wa = rng.random(40)
        # the negated row, hit 24 times with weights summing to sum(wa) (up to rounding)
        wb = rng.random(24)
        wb = wb / wb.sum() * wa.sum()
        other = rng.integers(0, 256, 6)
        idx.append(np.r_[np.full(40, r), np.full(24, r + 128), other])
        wts.append(np.r_[wa, wb, rng.random(6) * 1e-3])
    ind = torch.tensor(np.concatenate(idx), dtype=torch.int64)
    off = torch.arange(0, 70 * B + 1, 70, dtype=torch.int64)
    w = torch.tensor(np.concatenate(wts), dtype=torch.float32)
    for pooling in ("sum", "mean"):
        out, _ = run_hist(tables, ind, off, B, w, pooling)
        check_hist(out, tables, ind, off, B, w, pooling, what=f"cancelling {pooling}")


def test_histogram_bf16_values_below_fp16_normal_range():
    """bf16 tables whose values sit far below fp16's smallest normal (2^-14):
    the table-wide power-of-two scale brings them into range, exactly."""
    g = torch.Generator().manual_seed(25)
    for mag in (1e-7, 1e-20, 1e-30):
        tables = [(torch.randn((200, 32), generator=g) * mag).bfloat16().to(DEV)]
        B = 180
        ind, off = batch_for(200, B, 50, seed=26)
        w = torch.rand(ind.numel(), generator=g)
        out, paths = run_hist(tables, ind, off, B, w, "mean")
        assert paths == ["histogram"]
        ref = check_hist(out, tables, ind, off, B, w, "mean", what=f"bf16 tiny {mag}")
        assert np.abs(ref).max() > 0
        # the allowance is relative to the terms: at these magnitudes the
        # absolute floor alone would accept zeros, so check relative error too
        got = out.cpu().numpy()
        abs_sum, n = pooled_abs_sum(tables, ind, off, B, w, "mean")
        nz = abs_sum > 0
        rel = np.abs(got[nz] - ref[nz]) / abs_sum[nz]
        assert rel.max() < 2.0 ** -18, rel.max()


def test_histogram_small_weights_stay_accurate():
    """Weights of 1e-6 on fp16 rows of magnitude 100: without the per-bag
    scale the H entries would sit in fp16's subnormal range."""
    g = torch.Generator().manual_seed(27)
    tables = [(torch.randn((300, 48), generator=g) * 100.0).half().to(DEV)]
    B = 200
    ind, off = batch_for(300, B, 60, seed=28)
    w = torch.rand(ind.numel(), generator=g) * 1e-6
    out, _ = run_hist(tables, ind, off, B, w)
    check_hist(out, tables, ind, off, B, w, what="small weights")
    got = out.cpu().numpy()
    ref, _ = oracle_forward(tables, ind, off, B, w)
    abs_sum, _ = pooled_abs_sum(tables, ind, off, B, w)
    nz = abs_sum > 0
    assert (np.abs(got[nz] - ref[nz]) / abs_sum[nz]).max() < 2.0 ** -18


def test_histogram_large_scales_stay_on_the_tensor_cores():
    """Weights of 32768 on bags that repeat rows: an H entry (the sum of a
    bag's scales of one row) passes fp16's 65504; the per-bag scale keeps it
    in range, so every tile stays on the tensor cores at fp32 accuracy."""
    g = torch.Generator().manual_seed(11)
    tables = [(torch.randn((256, 32), generator=g) * 0.01).half().to(DEV)]
    B = 400
    rng = np.random.default_rng(12)
    lens = rng.integers(1, 40, B)
    idx = []
    for b in range(B):
        if b < 128:  # rows drawn from 4, so repeats
            idx.append(rng.integers(0, 4, lens[b]))
        else:  # distinct rows in each bag
            idx.append(rng.permutation(256)[:lens[b]])
    ind = torch.tensor(np.concatenate(idx), dtype=torch.int64)
    off = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int64)
    w = torch.full((ind.numel(),), 32768.0)
    out, paths = run_hist(tables, ind, off, B, w)
    assert paths == ["histogram"]
    check_hist(out, tables, ind, off, B, w, what="large scales")


def test_histogram_bf16_table_beyond_fp16_range():
    """A bf16 table holding a value of 1e6 (past fp16's 65504) next to values
    of 0.01: the table-wide scale brings the largest into range and keeps the
    others exact (they lie within 2^29 of it)."""
    g = torch.Generator().manual_seed(13)
    t = torch.randn((128, 16), generator=g) * 0.01
    t[5, 3] = 1.0e6
    tables = [t.bfloat16().to(DEV)]
    B = 200
    ind, off = batch_for(128, B, 30, seed=14)
    out, paths = run_hist(tables, ind, off, B, None, "mean")
    assert paths == ["histogram"]
    check_hist(out, tables, ind, off, B, None, "mean", what="hist bf16 beyond fp16")


def test_histogram_nonfinite_inputs_take_the_fp32_gather():
    """An inf weight makes its tile's outputs non-finite on the tensor cores;
    that tile is pooled again by the fp32 gather, so inf and NaN land where
    the oracle puts them."""
    g = torch.Generator().manual_seed(15)
    tables = [(torch.randn((128, 32), generator=g) * 0.01).half().to(DEV)]
    B = 200
    ind, off = batch_for(128, B, 30, seed=16)
    w = torch.rand(ind.numel(), generator=g)
    bag = next(b for b in range(70, B) if int(off[b + 1]) > int(off[b]))
    w[int(off[bag])] = float("inf")  # the first lookup of a non-empty bag
    out, _ = run_hist(tables, ind, off, B, w)
    ref, _ = oracle_forward(tables, ind, off, B, w)
    got = out.cpu().numpy()
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    np.testing.assert_array_equal(np.isinf(got), np.isinf(ref))
    fin = np.isfinite(ref)
    assert_close(got[fin], ref[fin], what="finite outputs", **FP32_TOL)


def test_histogram_long_bags_overflow_the_clear_lists():
    """Bags of up to 400 lookups: a warp's four bags then hold far more
    lookups than its registers (128) and its clear list (256) cover, so the
    chunks past the registers and the whole-slab clear both run."""
    g = torch.Generator().manual_seed(17)
    tables = [(torch.randn((512, 64), generator=g) * 0.01).half().to(DEV),
              (torch.randn((160, 32), generator=g) * 0.01).bfloat16().to(DEV)]
    B = 300
    i0, o0 = batch_for(512, B, 400, seed=18)
    i1, o1 = batch_for(160, B, 400, seed=19)
    ind = torch.cat([i0, i1])
    off = torch.cat([o0, o1[1:] + o0[-1]])
    w = torch.rand(ind.numel(), generator=g)
    out, paths = run_hist(tables, ind, off, B, w, "mean")
    assert paths == ["histogram", "histogram"]
    check_hist(out, tables, ind, off, B, w, "mean", what="long bags")


def test_histogram_tables_of_several_shapes_in_one_launch():
    """Four fp16 tables of different row counts and dims, B large enough that
    persistent CTAs cross from one table to the next (A is laid out again and
    W^T reloaded); two of the tables have ragged row counts."""
    g = torch.Generator().manual_seed(31)
    shapes = [(512, 64), (100, 16), (37, 48), (250, 32)]
    tables = [(torch.randn(s, generator=g) * 0.01).half().to(DEV) for s in shapes]
    B = 6000
    parts = [batch_for(r, B, 40, seed=32 + k) for k, (r, _) in enumerate(shapes)]
    ind = torch.cat([p[0] for p in parts])
    offs = [parts[0][1]]
    for p in parts[1:]:
        offs.append(p[1][1:] + offs[-1][-1])
    off = torch.cat(offs)
    w = torch.rand(ind.numel(), generator=g)
    out, paths = run_hist(tables, ind, off, B, w)
    assert paths == ["histogram"] * 4
    check_hist(out, tables, ind, off, B, w, what="several shapes")


def test_histogram_is_deterministic():
    """Entries are summed in a fixed order by the one warp that owns them, so
    two calls give bit-identical outputs."""
    g = torch.Generator().manual_seed(33)
    tables = [(torch.randn((512, 64), generator=g) * 0.01).half().to(DEV)]
    B = 3000
    ind, off = batch_for(512, B, 64, seed=34)
    ind = torch.tensor(np.random.default_rng(35).integers(0, 8, ind.numel()), dtype=torch.int64)  # many repeats
    w = torch.rand(ind.numel(), generator=g)
    h = tbe.tbe_create(tables, "sum", tbe.TBE_FLAG_FORCE_HISTOGRAM)
    a = tbe.tbe_forward(h, ind.to(DEV), off.to(DEV), B, w.to(DEV)).cpu()
    b = tbe.tbe_forward(h, ind.to(DEV), off.to(DEV), B, w.to(DEV)).cpu()
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    h.close()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    check_hist(a, tables, ind, off, B, w, what="repeats")


def test_histogram_out_of_range_and_int32():
    g = torch.Generator().manual_seed(3)
    tables = [(torch.randn((64, 32), generator=g) * 0.01).half().to(DEV),
              (torch.randn((5000, 32), generator=g) * 0.01).to(DEV)]
    B = 130
    i0, o0 = batch_for(64, B, 40, seed=4, oob=True)
    i1, o1 = batch_for(5000, B, 40, seed=5)
    ind = torch.cat([i0, i1]).to(torch.int32)
    off = torch.cat([o0, o1[1:] + o0[-1]]).to(torch.int32)
    out, paths = run_hist(tables, ind, off, B, expect=tbe.TBE_ERR_INDEX_OOB)
    assert paths == ["histogram", "gather"]
    ref, skipped = oracle_forward(tables, ind, off, B)
    assert skipped > 0
    assert_close(out.cpu().numpy(), ref, what="hist oob", **FP32_TOL)


def test_histogram_workload_small_tables():
    """The 64 fp16 512x64 tables plus one large fp32 table, B shrunk: the small
    tables run on the histogram path, the large one on the gather path."""
    cfg = workloads.get_config(5).scaled(B=300, rows_div=1000, rows_min=512)
    specs = workloads.realize_tables(cfg)
    tables = [t.to(DEV) for t in workloads.make_tables(cfg, "cpu", specs)]
    batch = workloads.make_batch(cfg, "cpu", torch.int64, specs)
    h = tbe.tbe_create(tables, cfg.pooling, tbe.TBE_FLAG_FORCE_HISTOGRAM)
    paths = tbe.tbe_table_paths(h)
    assert paths[:64] == ["histogram"] * 64 and paths[64] == "gather"
    out = tbe.tbe_forward(h, batch.indices.to(DEV), batch.offsets.to(DEV), cfg.B, batch.weights.to(DEV))
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    h.close()
    check_hist(out, tables, batch.indices, batch.offsets, cfg.B, batch.weights, cfg.pooling,
               what="hist tables", cols=slice(0, 64 * 64))
    ref, _ = oracle_forward(tables, batch.indices, batch.offsets, cfg.B, batch.weights, cfg.pooling)
    assert_close(out.cpu().numpy()[:, 64 * 64:], ref[:, 64 * 64:], what="gather table", **FP32_TOL)


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


def test_dense_backward_forced_1024_rows():
    """TBE_FLAG_FORCE_HISTOGRAM admits tables of up to 1024 rows to the dense
    backward: at dim 128 a table spans four row groups of CTAs (two 128-row
    M tiles each), next to a 1000 x 64 table and a sorted-path table."""
    specs = [(1024, 128, torch.bfloat16), (1000, 64, torch.float16), (4000, 32, torch.float32)]
    _dense_case(specs, 200, "sum", True, "sgd", flags=tbe.TBE_FLAG_FORCE_HISTOGRAM, seed=31)


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


@pytest.mark.parametrize("pooling,weighted", [("sum", True), ("mean", False)])
def test_histogram_forward_with_length_order(pooling, weighted):
    """TBE_FLAG_LENGTH_ORDER and the histogram forward on one handle (the
    order applies to the gathered tables; the histogram tiles keep index
    order).  Lengths 0..90 (empty bags included), several tables of both
    16-bit dtypes, B not a multiple of the 64-bag tile: the result matches
    the oracle within the histogram allowance, with and without the flag."""
    g = torch.Generator().manual_seed(21)
    specs = [(512, 64, torch.float16), (300, 32, torch.float16), (512, 64, torch.bfloat16)]
    tables = [(torch.randn((r, d), generator=g) * 0.01).to(dt).to(DEV) for r, d, dt in specs]
    B = 1000
    rng = np.random.default_rng(22)
    lengths = rng.integers(0, 91, len(specs) * B)
    ind = torch.tensor(np.concatenate([rng.integers(0, specs[t][0], lengths[t * B + b])
                                       for t in range(len(specs)) for b in range(B)]), dtype=torch.int64)
    off = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int64)
    w = torch.rand(ind.numel(), generator=g) if weighted else None
    flags = tbe.TBE_FLAG_FORCE_HISTOGRAM
    out_o, paths = run_hist(tables, ind, off, B, w, pooling, flags | tbe.TBE_FLAG_LENGTH_ORDER)
    assert paths == ["histogram"] * 3
    out_i, _ = run_hist(tables, ind, off, B, w, pooling, flags)
    check_hist(out_o, tables, ind, off, B, w, pooling, what="histogram, length order")
    check_hist(out_i, tables, ind, off, B, w, pooling, what="histogram, index order")
