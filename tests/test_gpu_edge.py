"""GPU parity on edge cases and path switches: run lengths around the 256
threshold and far above it, applying a prepared workspace twice, empty and
ragged batches, bags long enough for the CTA path, element-wise dims,
unaligned tables, mixed table classes in one handle, and the device error
flags (out-of-range indices, malformed offsets)."""

import numpy as np
import pytest
import torch

import oracle
import recommender_sparse_embeddings_gb300 as tbe
from helpers import (FP32_TOL, DT_NAME, assert_close, assert_tables_match, oracle_backward,
                     oracle_forward, table_bits, touched_rows)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def make_tables(specs, seed=0):
    """specs: list of (rows, dim, torch dtype)."""
    g = torch.Generator().manual_seed(seed)
    return [(torch.randn((r, d), generator=g) * 0.01).to(dt).to(DEV) for r, d, dt in specs]


def csr(bags_per_table, index_dtype=torch.int64):
    """bags_per_table: list (per table) of lists (per bag) of row indices."""
    B = len(bags_per_table[0])
    assert all(len(b) == B for b in bags_per_table)
    lengths = [len(bag) for tab in bags_per_table for bag in tab]
    flat = [i for tab in bags_per_table for bag in tab for i in bag]
    ind = torch.tensor(flat, dtype=index_dtype)
    off = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=index_dtype)
    return ind, off, B


def run_backward_and_compare(tables, ind, off, B, grad, optimizer, lr=0.01, eps=1e-8, weights=None,
                             pooling="sum", what=""):
    cpu_tables = [t.cpu() for t in tables]
    before = [table_bits(t) for t in tables]
    h = tbe.tbe_create(tables, pooling)
    ws = tbe.make_workspace(h, ind.numel(), B)
    w = None if weights is None else weights.to(DEV)
    total_rows = sum(t.shape[0] for t in tables)
    state = None
    if optimizer == "sgd":
        tbe.tbe_backward_sgd(h, ind.to(DEV), off.to(DEV), B, grad.to(DEV), lr, ws, w)
    else:
        state = torch.zeros(total_rows, dtype=torch.float32, device=DEV)
        tbe.tbe_backward_rowwise_adagrad(h, ind.to(DEV), off.to(DEV), B, grad.to(DEV), state, lr, eps, ws, w)
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    ref_tabs, ref_state = oracle_backward(cpu_tables, ind, off, B, grad, optimizer, lr, eps, weights, pooling,
                                          None if state is None else torch.zeros(total_rows))
    touched = touched_rows(cpu_tables, ind, off, B)
    assert_tables_match(tables, ref_tabs, before, touched, what=what)
    if state is not None:
        assert_close(state.cpu().numpy(), ref_state, what=f"{what} state", **FP32_TOL)
    h.close()


@pytest.mark.parametrize("optimizer", ["sgd", "adagrad"])
@pytest.mark.parametrize("dtype,dim", [(torch.float32, 128), (torch.bfloat16, 64), (torch.float16, 256),
                                       (torch.float32, 32)])
def test_run_length_threshold(optimizer, dtype, dim):
    """Rows hit exactly 1, 255, 256, 257, 512 and 100000 times."""
    rng = np.random.default_rng(7)
    R, B = 1000, 4096
    counts = {3: 1, 10: 255, 11: 256, 12: 257, 20: 512, 30: 100000}
    lookups = np.concatenate([np.full(c, r) for r, c in counts.items()])
    rng.shuffle(lookups)
    cuts = np.sort(rng.choice(np.arange(1, len(lookups)), size=B - 1, replace=False))
    bags = [list(map(int, x)) for x in np.split(lookups, cuts)]
    ind, off, B = csr([bags])
    tables = make_tables([(R, dim, dtype)], seed=1)
    grad = torch.randn((B, dim), generator=torch.Generator().manual_seed(2))
    run_backward_and_compare(tables, ind, off, B, grad, optimizer, what=f"threshold {dtype} {dim}")


@pytest.mark.parametrize("optimizer", ["sgd", "adagrad"])
def test_sparse_batch_bag_ids_beyond_the_lookup_count(optimizer):
    """Without per-lookup scales the sort carries each lookup's flat bag,
    and a flat bag id can exceed the number of lookups: here 2 x 6000 bags
    hold 700 lookups, all in bags past id 700 (the second table's bags are
    5999 and up), one row hit 400 times (a long run) and others once."""
    rng = np.random.default_rng(17)
    B = 6000
    tabs = [[[] for _ in range(B)] for _ in range(2)]
    for k in range(400):  # table 0: row 5 in bags 1000..1399, a long run
        tabs[0][1000 + k].append(5)
    for b in rng.choice(np.arange(2000, B), size=150, replace=False):
        tabs[0][int(b)].append(int(rng.integers(0, 900)))
    for b in rng.choice(np.arange(0, B), size=150, replace=False):
        tabs[1][int(b)].append(int(rng.integers(0, 700)))
    ind, off, B = csr(tabs)
    assert ind.numel() == 700 and 2 * B > 8 * ind.numel()
    tables = make_tables([(900, 128, torch.float32), (700, 64, torch.bfloat16)], seed=18)
    grad = torch.randn((B, 192), generator=torch.Generator().manual_seed(19))
    run_backward_and_compare(tables, ind, off, B, grad, optimizer, what=f"sparse batch {optimizer}")


def test_prepared_workspace_applies_twice():
    """prepare once, apply twice (the long-run completion counts reset)."""
    rng = np.random.default_rng(3)
    R, B, D = 500, 512, 128
    bags = [list(map(int, rng.choice(np.r_[np.zeros(40, int), rng.integers(0, R, 40)], 8))) for _ in range(B)]
    ind, off, B = csr([bags])
    tables = make_tables([(R, D, torch.float32)], seed=4)
    cpu_tables = [t.cpu() for t in tables]
    grad = torch.randn((B, D), generator=torch.Generator().manual_seed(5))
    h = tbe.tbe_create(tables, "sum")
    ws = tbe.make_workspace(h, ind.numel(), B)
    tbe.tbe_backward_prepare(h, ind.to(DEV), off.to(DEV), B, ws)
    for _ in range(2):
        tbe.tbe_backward_apply(h, ind.numel(), B, grad.to(DEV), ws, "sgd", 0.05)
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    tabs = [table_bits(t) for t in cpu_tables]
    for _ in range(2):
        oracle.backward(tabs, ["f32"], ind.numpy(), off.numpy(), B, grad.numpy(), "sgd", 0.05)
    assert_close(tables[0].cpu().numpy(), tabs[0], what="two applies", **FP32_TOL)
    h.close()


@pytest.mark.parametrize("index_dtype", [torch.int64, torch.int32])
def test_mixed_classes_empty_bags_and_weights(index_dtype):
    """One handle: fp32 d128, bf16 d32, fp16 d64 (vector classes), fp32 d3,
    bf16 d12, fp32 d1 (element-wise); many empty bags; weights; mean and sum
    pooling."""
    rng = np.random.default_rng(11)
    specs = [(300, 128, torch.float32), (50, 32, torch.bfloat16), (70, 64, torch.float16),
             (40, 3, torch.float32), (90, 12, torch.bfloat16), (25, 1, torch.float32)]
    B = 333
    bags = []
    for r, _, _ in specs:
        lens = rng.integers(0, 9, B)
        lens[rng.random(B) < 0.3] = 0
        bags.append([list(map(int, rng.integers(0, r, n))) for n in lens])
    ind, off, B = csr(bags, index_dtype)
    w = torch.rand(ind.numel(), generator=torch.Generator().manual_seed(3))
    total_d = sum(d for _, d, _ in specs)
    for pooling in ("sum", "mean"):
        tables = make_tables(specs, seed=5)
        h = tbe.tbe_create(tables, pooling, tbe.TBE_FLAG_NO_HISTOGRAM)
        out = tbe.tbe_forward(h, ind.to(DEV), off.to(DEV), B, w.to(DEV))
        assert tbe.tbe_get_error(h) == tbe.TBE_OK
        ref, _ = oracle_forward(tables, ind, off, B, w, pooling)
        assert_close(out.cpu().numpy(), ref, what=f"forward {pooling}", **FP32_TOL)
        h.close()
        grad = torch.randn((B, total_d), generator=torch.Generator().manual_seed(6))
        run_backward_and_compare(tables, ind, off, B, grad, "adagrad", weights=w, pooling=pooling,
                                 what=f"mixed {pooling}")


def test_empty_batch_and_single_bag():
    tables = make_tables([(10, 16, torch.float32)])
    h = tbe.tbe_create(tables, "mean")
    B = 5
    ind = torch.zeros(0, dtype=torch.int64, device=DEV)
    off = torch.zeros(B + 1, dtype=torch.int64, device=DEV)
    out = tbe.tbe_forward(h, ind, off, B)
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    assert (out == 0).all()
    ws = tbe.make_workspace(h, 0, B)
    before = tables[0].clone()
    tbe.tbe_backward_sgd(h, ind, off, B, torch.ones((B, 16), device=DEV), 0.1, ws)
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    assert torch.equal(before, tables[0])
    h.close()
    ind, off, B = csr([[[2, 2, 7]]])
    run_backward_and_compare(tables, ind, off, B, torch.ones((1, 16)), "sgd", what="single bag")


@pytest.mark.parametrize("dtype,dim", [(torch.float32, 128), (torch.bfloat16, 256), (torch.float32, 7)])
def test_long_bags_take_the_cta_path(dtype, dim):
    """Bags of 3000 and 70000 lookups (beyond the per-slot limit) next to short ones."""
    rng = np.random.default_rng(8)
    R = 5000
    lens = [3000, 4, 70000, 0, 17, 2049]
    bags = [list(map(int, rng.integers(0, R, n))) for n in lens]
    ind, off, B = csr([bags])
    w = torch.rand(ind.numel(), generator=torch.Generator().manual_seed(1))
    tables = make_tables([(R, dim, dtype)], seed=9)
    for pooling in ("sum", "mean"):
        h = tbe.tbe_create(tables, pooling)
        for rep in range(2):  # the long-bag list alternates counters between calls
            out = tbe.tbe_forward(h, ind.to(DEV), off.to(DEV), B, w.to(DEV))
            assert tbe.tbe_get_error(h) == tbe.TBE_OK
            ref, _ = oracle_forward(tables, ind, off, B, w, pooling)
            assert_close(out.cpu().numpy(), ref, what=f"long bags {pooling} {rep}", **FP32_TOL)
        h.close()


def test_unaligned_table_uses_elementwise_paths():
    base = make_tables([(401, 128, torch.float32)], seed=12)[0]
    table = base.view(-1)[1:1 + 400 * 128].view(400, 128)  # 4-byte offset: not 16-byte aligned
    assert table.data_ptr() % 16 != 0
    h = tbe.tbe_create([table], "sum")
    assert tbe.tbe_table_paths(h) == ["gather_elementwise"]
    h.close()
    rng = np.random.default_rng(13)
    bags = [list(map(int, rng.integers(0, 400, rng.integers(0, 6)))) for _ in range(100)]
    ind, off, B = csr([bags])
    h = tbe.tbe_create([table], "sum")
    out = tbe.tbe_forward(h, ind.to(DEV), off.to(DEV), B)
    ref, _ = oracle_forward([table], ind, off, B)
    assert_close(out.cpu().numpy(), ref, what="unaligned forward", **FP32_TOL)
    h.close()
    grad = torch.randn((B, 128), generator=torch.Generator().manual_seed(14))
    run_backward_and_compare([table], ind, off, B, grad, "adagrad", what="unaligned backward")


def test_out_of_range_indices_are_skipped_and_reported():
    tables = make_tables([(50, 64, torch.float32), (30, 32, torch.bfloat16)], seed=15)
    bags = [[[1, 2, -1, 49], [50, 3], []], [[0, 29, 30], [1000], [5]]]
    ind, off, B = csr(bags)
    h = tbe.tbe_create(tables, "sum", tbe.TBE_FLAG_NO_HISTOGRAM)
    out = tbe.tbe_forward(h, ind.to(DEV), off.to(DEV), B)
    assert tbe.tbe_get_error(h) == tbe.TBE_ERR_INDEX_OOB
    assert tbe.tbe_get_error(h) == tbe.TBE_OK  # reading clears the flag
    ref, skipped = oracle_forward(tables, ind, off, B)
    assert skipped == 4
    assert_close(out.cpu().numpy(), ref, what="oob forward", **FP32_TOL)
    cpu_tables = [t.cpu() for t in tables]
    before = [table_bits(t) for t in tables]
    grad = torch.randn((B, 96), generator=torch.Generator().manual_seed(16))
    ws = tbe.make_workspace(h, ind.numel(), B)
    tbe.tbe_backward_sgd(h, ind.to(DEV), off.to(DEV), B, grad.to(DEV), 0.1, ws)
    assert tbe.tbe_get_error(h) == tbe.TBE_ERR_INDEX_OOB
    ref_tabs, _ = oracle_backward(cpu_tables, ind, off, B, grad, "sgd", 0.1)
    assert_tables_match(tables, ref_tabs, before, touched_rows(cpu_tables, ind, off, B), what="oob backward")
    h.close()


def test_malformed_offsets_are_reported():
    """Offsets that decrease (all values inside [0, N]) raise BAD_OFFSETS."""
    tables = make_tables([(20, 16, torch.float32)])
    h = tbe.tbe_create(tables, "sum")
    ind = torch.tensor([1, 2, 3, 4, 5, 6], dtype=torch.int64, device=DEV)
    off = torch.tensor([0, 4, 2, 6], dtype=torch.int64, device=DEV)
    tbe.tbe_forward(h, ind, off, 3)
    assert tbe.tbe_get_error(h) == tbe.TBE_ERR_BAD_OFFSETS
    ws = tbe.make_workspace(h, 6, 3)
    tbe.tbe_backward_sgd(h, ind, off, 3, torch.zeros((3, 16), device=DEV), 0.1, ws)
    assert tbe.tbe_get_error(h) == tbe.TBE_ERR_BAD_OFFSETS
    h.close()


def test_malformed_offsets_on_a_histogram_table_are_reported():
    """The same decreasing offsets on a small fp16 table: the histogram forward
    and the dense backward report BAD_OFFSETS (every read stays inside the
    batch: offsets are clamped to [0, N])."""
    tables = make_tables([(64, 16, torch.float16)])
    h = tbe.tbe_create(tables, "sum", tbe.TBE_FLAG_FORCE_HISTOGRAM)
    assert tbe.tbe_table_paths(h) == ["histogram"]
    assert tbe.tbe_backward_paths(h) == ["dense"]
    ind = torch.tensor([1, 2, 3, 4, 5, 6], dtype=torch.int64, device=DEV)
    off = torch.tensor([0, 4, 2, 6], dtype=torch.int64, device=DEV)
    tbe.tbe_forward(h, ind, off, 3)
    assert tbe.tbe_get_error(h) == tbe.TBE_ERR_BAD_OFFSETS
    ws = tbe.make_workspace(h, 6, 3)
    tbe.tbe_backward_sgd(h, ind, off, 3, torch.zeros((3, 16), device=DEV), 0.1, ws)
    assert tbe.tbe_get_error(h) == tbe.TBE_ERR_BAD_OFFSETS
    h.close()


def test_workspace_too_small_is_rejected_before_launch():
    tables = make_tables([(20, 16, torch.float32)])
    h = tbe.tbe_create(tables, "sum")
    ind = torch.tensor([1, 2], dtype=torch.int64, device=DEV)
    off = torch.tensor([0, 2], dtype=torch.int64, device=DEV)
    small = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(tbe.TBEError) as e:
        tbe.tbe_backward_sgd(h, ind, off, 1, torch.ones((1, 16), device=DEV), 0.1, small)
    assert e.value.code == tbe.TBE_ERR_WORKSPACE_TOO_SMALL
    h.close()


@pytest.mark.parametrize("cid", [2, 3])
def test_forward_prepare_side_by_side(cid):
    """tbe_forward_prepare (forward and preparation on two streams) gives the
    forward output, sort and run-length results, and after apply the tables,
    of the separate calls and the oracle."""
    import workloads
    cfg = workloads.get_config(cid).scaled(B=200, rows_div=1000, rows_min=64)
    specs = workloads.realize_tables(cfg)
    tables = [t.to(DEV) for t in workloads.make_tables(cfg, "cpu", specs)]
    batch = workloads.make_batch(cfg, "cpu", torch.int64, specs)
    grad = workloads.make_grad(cfg, "cpu", specs)
    cpu_tables = [t.cpu() for t in tables]
    before = [table_bits(t) for t in tables]
    h = tbe.tbe_create(tables, cfg.pooling, tbe.TBE_FLAG_NO_HISTOGRAM)
    ind, off = batch.indices.to(DEV), batch.offsets.to(DEV)
    w = None if batch.weights is None else batch.weights.to(DEV)
    ws = tbe.make_workspace(h, batch.N, cfg.B)
    out = tbe.tbe_forward_prepare(h, ind, off, cfg.B, ws, w)
    state = torch.zeros(h.total_rows, dtype=torch.float32, device=DEV) if cfg.optimizer == "adagrad" else None
    tbe.tbe_backward_apply(h, batch.N, cfg.B, grad.to(DEV), ws, cfg.optimizer, cfg.lr, cfg.eps, state)
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    ref, _ = oracle_forward(cpu_tables, batch.indices, batch.offsets, cfg.B, batch.weights, cfg.pooling)
    assert_close(out.cpu().numpy(), ref, what="fused forward", **FP32_TOL)
    lay = tbe.tbe_backward_workspace_layout(h, batch.N, cfg.B)
    keys, _ = oracle.make_keys([t.shape[0] for t in cpu_tables], batch.indices.numpy(), batch.offsets.numpy(), cfg.B)
    r = oracle.sort_rle(keys)
    got = ws[lay.sorted_keys:lay.sorted_keys + 4 * batch.N].view(torch.int32).cpu().numpy().view(np.uint32)
    np.testing.assert_array_equal(got.astype(np.int64), r["sorted_keys"])
    ref_tabs, ref_state = oracle_backward(cpu_tables, batch.indices, batch.offsets, cfg.B, grad, cfg.optimizer,
                                          cfg.lr, cfg.eps, batch.weights, cfg.pooling,
                                          None if state is None else torch.zeros(h.total_rows))
    assert_tables_match(tables, ref_tabs, before, touched_rows(cpu_tables, batch.indices, batch.offsets, cfg.B),
                        what="fused then apply")
    if state is not None:
        assert_close(state.cpu().numpy(), ref_state, what="fused state", **FP32_TOL)
    h.close()
