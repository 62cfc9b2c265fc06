"""tbe_backward_sgd_noalloc: backward + SGD for callers that cannot allocate.

Some callers cannot call cudaMalloc when they run the backward pass, because
another allocator owns their device memory (a framework's caching allocator
has reserved it, or a fixed pool was handed out at start-up), or because they
forbid device allocation once set-up is over.  They cannot supply the
workspace tbe_backward_sgd asks for.  The no-alloc entry point runs the same
kernels on a 32 MiB static device array inside the library instead.

The tests call it through the C ABI and check its updated tables against
those of tbe_backward_sgd (with a workspace of its own) on identical copies of
the inputs, for two calls in a row; a second test first runs it on a
different batch (more lookups, weights, another handle with histogram
tables), so the static array holds that call's leftovers, then checks the
next call bit for bit against tbe_backward_sgd and against the CPU oracle.
They live in a file of their own that pytest collects last, and they work in
a fresh process as well as after the other tests.
"""

import ctypes

import pytest
import torch

import recommender_sparse_embeddings_gb300 as tbe
import workloads
from helpers import (FP32_TOL, LOWP_TOL, DT_NAME, assert_close, assert_tables_match, decoded, oracle_backward,
                     table_bits, touched_rows)

pytestmark = pytest.mark.gpu

DEV = "cuda"
STATIC_SCRATCH_BYTES = 32 << 20


def _noalloc_call(lib, h, ind, off, B, grad, lr, weights=None):
    """Direct C-ABI call (no binding helper, no allocation in between)."""
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.tbe_backward_sgd_noalloc(
        h.ptr, ctypes.c_void_p(ind.data_ptr()), ctypes.c_void_p(off.data_ptr()),
        tbe.TBE_I64 if ind.dtype == torch.int64 else tbe.TBE_I32, ind.numel(), B,
        None if weights is None else ctypes.c_void_p(weights.data_ptr()),
        ctypes.c_void_p(grad.data_ptr()), ctypes.c_float(lr), stream)


@pytest.mark.parametrize("cid,B,rows_div,rows_min", [(1, 64, 1, 1), (2, 300, 1000, 64), (5, 96, 1000, 512)])
def test_noalloc_matches_workspace_entry_point_twice(cid, B, rows_div, rows_min):
    lib = tbe.load_library()
    cfg = workloads.get_config(cid)
    if (B, rows_div) != (cfg.B, 1):
        cfg = cfg.scaled(B=B, rows_div=rows_div, rows_min=rows_min)
    specs = workloads.realize_tables(cfg)
    base = [t.to(DEV) for t in workloads.make_tables(cfg, "cpu", specs)]
    tabs_a = [t.clone() for t in base]  # tbe_backward_sgd with its own workspace
    tabs_b = [t.clone() for t in base]  # tbe_backward_sgd_noalloc
    h_a = tbe.tbe_create(tabs_a, cfg.pooling)
    h_b = tbe.tbe_create(tabs_b, cfg.pooling)
    batch = workloads.make_batch(cfg, DEV, torch.int64, specs)
    grad = workloads.make_grad(cfg, DEV, specs)
    assert tbe.tbe_backward_workspace_bytes(h_b, batch.N, cfg.B) <= STATIC_SCRATCH_BYTES
    ws = tbe.make_workspace(h_a, batch.N, cfg.B)
    for step in range(2):
        tbe.tbe_backward_sgd(h_a, batch.indices, batch.offsets, cfg.B, grad, cfg.lr, ws,
                             batch.weights)
        rc = _noalloc_call(lib, h_b, batch.indices, batch.offsets, cfg.B, grad, cfg.lr, batch.weights)
        assert rc == tbe.TBE_OK, tbe.tbe_strerror(rc)
        assert tbe.tbe_get_error(h_a) == tbe.TBE_OK
        assert tbe.tbe_get_error(h_b) == tbe.TBE_OK
        for t, (a, b) in enumerate(zip(tabs_a, tabs_b)):
            tol = FP32_TOL if a.dtype == torch.float32 else LOWP_TOL
            assert_close(decoded(b), decoded(a), what=f"step {step} table {t}", **tol)
    h_a.close()
    h_b.close()


def test_noalloc_rejects_batches_beyond_its_scratch():
    lib = tbe.load_library()
    table = torch.zeros((1000, 128), dtype=torch.float32, device=DEV)
    h = tbe.tbe_create([table], "sum")
    N, B = 2_000_000, 1000
    assert tbe.tbe_backward_workspace_bytes(h, N, B) > STATIC_SCRATCH_BYTES
    ind = torch.zeros(N, dtype=torch.int64, device=DEV)
    off = torch.arange(0, N + 1, N // B, dtype=torch.int64, device=DEV)
    grad = torch.ones((B, 128), dtype=torch.float32, device=DEV)
    torch.cuda.synchronize()
    rc = _noalloc_call(lib, h, ind, off, B, grad, 0.5)
    assert rc == tbe.TBE_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert not table.any()  # nothing ran
    h.close()


def test_noalloc_leftovers_of_another_batch_do_no_harm():
    lib = tbe.load_library()
    # 1. fill the static array with another call's state: a handle with a
    #    histogram table (dense backward), a weighted batch of more lookups
    g = torch.Generator().manual_seed(71)
    other = [(torch.randn((512, 64), generator=g) * 0.01).half().to(DEV),
             (torch.randn((40000, 32), generator=g) * 0.01).to(DEV),
             (torch.randn((3000, 128), generator=g) * 0.01).bfloat16().to(DEV)]
    B1 = 700
    lens = torch.randint(0, 90, (3 * B1,), generator=g)
    off1 = torch.cat([torch.zeros(1, dtype=torch.int64), lens.cumsum(0)])
    N1 = int(off1[-1])
    rows = torch.tensor([512, 40000, 3000]).repeat_interleave(lens.view(3, B1).sum(1))
    ind1 = (torch.rand(N1, generator=g) * rows).to(torch.int64)
    w1 = torch.rand(N1, generator=g)
    grad1 = torch.randn((B1, 224), generator=g)
    h1 = tbe.tbe_create(other, "mean")
    assert tbe.tbe_backward_workspace_bytes(h1, N1, B1) <= STATIC_SCRATCH_BYTES
    rc = _noalloc_call(lib, h1, ind1.to(DEV), off1.to(DEV), B1, grad1.to(DEV), 0.05, w1.to(DEV))
    assert rc == tbe.TBE_OK, tbe.tbe_strerror(rc)
    assert tbe.tbe_get_error(h1) == tbe.TBE_OK
    h1.close()

    # 2. the checked call: fewer lookups, no weights, sum pooling, a handle
    #    with another table layout (sorted backward only, deterministic)
    cfg = workloads.get_config(2).scaled(B=256, rows_div=1000, rows_min=64)
    specs = workloads.realize_tables(cfg)
    base = workloads.make_tables(cfg, "cpu", specs)
    batch = workloads.make_batch(cfg, "cpu", torch.int64, specs)
    grad = workloads.make_grad(cfg, "cpu", specs)
    assert batch.N < N1 and batch.weights is None
    tabs_a = [t.to(DEV) for t in base]
    tabs_b = [t.to(DEV) for t in base]
    h_a = tbe.tbe_create(tabs_a, cfg.pooling)
    h_b = tbe.tbe_create(tabs_b, cfg.pooling)
    ws = tbe.make_workspace(h_a, batch.N, cfg.B)
    ind, off, gd = batch.indices.to(DEV), batch.offsets.to(DEV), grad.to(DEV)
    tbe.tbe_backward_sgd(h_a, ind, off, cfg.B, gd, cfg.lr, ws)
    rc = _noalloc_call(lib, h_b, ind, off, cfg.B, gd, cfg.lr)
    assert rc == tbe.TBE_OK, tbe.tbe_strerror(rc)
    assert tbe.tbe_get_error(h_a) == tbe.TBE_OK
    assert tbe.tbe_get_error(h_b) == tbe.TBE_OK
    for t, (a, b) in enumerate(zip(tabs_a, tabs_b)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32)), f"table {t} differs from tbe_backward_sgd"
    # and directly against the oracle
    ref, _ = oracle_backward(base, batch.indices, batch.offsets, cfg.B, grad, "sgd", cfg.lr)
    before = [table_bits(t) for t in base]
    assert_tables_match(tabs_b, ref, before, touched_rows(base, batch.indices, batch.offsets, cfg.B),
                        what="noalloc vs oracle")
    h_a.close()
    h_b.close()
