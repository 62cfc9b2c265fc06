"""Bit-exact GPU parity: small-integer tables, power-of-two weights, integer
upstream gradients and a power-of-two learning rate make every sum and
product of the method exact in fp32 (all magnitudes stay far below 2^24), so
the result does not depend on the order of additions, and the CUDA path must
match the oracle bit for bit on every path: vector and element-wise
gathers, long bags, the histogram tensor-core forward, the sorted backward
(short and long runs) and the dense tensor-core backward.  The rounding of
an updated fp16/bf16 row is then the rounding of one exact value, the same
on both sides."""

import numpy as np
import pytest
import torch

import oracle
import recommender_sparse_embeddings_gb300 as tbe
from helpers import DT_NAME, table_bits

pytestmark = pytest.mark.gpu

DEV = "cuda"

# (rows, dim, dtype): vector gather (fp32 128, bf16 64), element-wise gather
# (fp32 dim 3), histogram tables (fp16 512 x 64, bf16 200 x 32)
SPECS = [(3000, 128, torch.float32), (900, 64, torch.bfloat16), (50, 3, torch.float32),
         (512, 64, torch.float16), (200, 32, torch.bfloat16)]


def integer_problem(seed, B, long_bag=False):
    rng = np.random.default_rng(seed)
    tables = [torch.from_numpy(rng.integers(-8, 9, (r, d)).astype(np.float32)).to(dt).to(DEV)
              for r, d, dt in SPECS]
    T = len(SPECS)
    lens = rng.integers(0, 40, T * B)
    if long_bag:
        lens[1] = 3000  # a bag of table 0 past the long-bag threshold
    idx = []
    for t, (r, _, _) in enumerate(SPECS):
        n = int(lens[t * B:(t + 1) * B].sum())
        hot = rng.integers(0, r, 4)
        ii = rng.integers(0, r, n)
        ii[rng.random(n) < 0.3] = hot[0]  # a row hit often enough for long runs
        idx.append(ii)
    ind = torch.from_numpy(np.concatenate(idx).astype(np.int64))
    off = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int64))
    w = torch.from_numpy(rng.choice([0.25, 0.5, 1.0, 2.0], ind.numel()).astype(np.float32))
    grad = torch.from_numpy(rng.integers(-4, 5, (B, sum(d for _, d, _ in SPECS))).astype(np.float32))
    return tables, ind, off, w, grad


@pytest.mark.parametrize("long_bag", [False, True])
@pytest.mark.parametrize("flags", [0, tbe.TBE_FLAG_FORCE_HISTOGRAM])
def test_forward_bit_exact(long_bag, flags):
    """Default flags: every table on the gather; with the histogram flag the
    two small tables on the tensor cores."""
    B = 300
    tables, ind, off, w, _ = integer_problem(1, B, long_bag)
    h = tbe.tbe_create(tables, "sum", flags)
    small = "histogram" if flags else "gather"
    assert tbe.tbe_table_paths(h) == ["gather", "gather", "gather_elementwise", small, small]
    out = tbe.tbe_forward(h, ind.to(DEV), off.to(DEV), B, w.to(DEV))
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    ref, skipped = oracle.forward([table_bits(t) for t in tables], [DT_NAME[t.dtype] for t in tables],
                                  ind.numpy(), off.numpy(), B, weights=w.numpy())
    assert skipped == 0
    np.testing.assert_array_equal(out.cpu().numpy(), ref)
    h.close()


@pytest.mark.parametrize("flags", [0, tbe.TBE_FLAG_SORTED_BACKWARD])
def test_sgd_backward_bit_exact(flags):
    """Default flags: the small tables take the dense backward; with
    TBE_FLAG_SORTED_BACKWARD every table takes the sort."""
    B = 300
    tables, ind, off, w, grad = integer_problem(2, B)
    before = [table_bits(t) for t in tables]
    h = tbe.tbe_create(tables, "sum", flags)
    ws = tbe.make_workspace(h, ind.numel(), B)
    tbe.tbe_backward_sgd(h, ind.to(DEV), off.to(DEV), B, grad.to(DEV), 0.5, ws, w.to(DEV))
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    ref = [b.copy() for b in before]
    oracle.backward(ref, [DT_NAME[t.dtype] for t in tables], ind.numpy(), off.numpy(), B, grad.numpy(), "sgd",
                    0.5, weights=w.numpy())
    for t, tab in enumerate(tables):
        np.testing.assert_array_equal(table_bits(tab), ref[t], err_msg=f"table {t}")
    h.close()


def test_cuda_graph_replay_matches_stream_launches():
    """The step (forward + preparation side by side, then SGD apply) captured
    as CUDA graphs and replayed gives the same bits as the same calls
    launched on a stream: the library's side streams fork from and join back
    into the capturing stream."""
    B = 300
    tables_a, ind, off, w, grad = integer_problem(3, B)
    tables_b = [t.clone() for t in tables_a]
    ind, off, w, grad = ind.to(DEV), off.to(DEV), w.to(DEV), grad.to(DEV)

    def step(h, ws, out, lr):
        tbe.tbe_forward_prepare(h, ind, off, B, ws, w, out)
        tbe.tbe_backward_apply(h, ind.numel(), B, grad, ws, "sgd", lr, 0.0, None)

    ha = tbe.tbe_create(tables_a, "sum")
    ws_a = tbe.make_workspace(ha, ind.numel(), B)
    out_a = torch.empty((B, ha.total_dim), dtype=torch.float32, device=DEV)
    step(ha, ws_a, out_a, 0.5)
    assert tbe.tbe_get_error(ha) == tbe.TBE_OK

    hb = tbe.tbe_create(tables_b, "sum")
    ws_b = tbe.make_workspace(hb, ind.numel(), B)
    out_b = torch.empty_like(out_a)
    step(hb, ws_b, out_b, 0.0)  # warm-up: lr 0 leaves the rows as they are
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(hb, ws_b, out_b, 0.5)
    out_b.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert tbe.tbe_get_error(hb) == tbe.TBE_OK
    np.testing.assert_array_equal(out_b.cpu().numpy(), out_a.cpu().numpy())
    for t in range(len(tables_a)):
        np.testing.assert_array_equal(table_bits(tables_b[t]), table_bits(tables_a[t]), err_msg=f"table {t}")
    ha.close()
    hb.close()
