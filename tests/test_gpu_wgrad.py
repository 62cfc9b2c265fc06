"""GPU parity of the per-sample weight gradient (tbe_per_sample_weight_grad)
against the oracle: dL/dw_i = (1/L if mean) <W_t[idx_i], G[b, cols of t]>,
0 for a skipped lookup.

Each output is a dot product of D fp32 products, so besides the fp32
tolerance every entry may differ by the rounding of that sum: four times
sqrt(D) * 2^-24 * sum_j |G_j W_j| (the same allowance the row sums get)."""

import numpy as np
import pytest
import torch

import oracle
import recommender_sparse_embeddings_gb300 as tbe
import workloads
from helpers import DT_NAME, FP32_TOL, accumulation_allowance, assert_close, table_bits
from test_gpu_parity import make_problem

pytestmark = pytest.mark.gpu

DEV = "cuda"
TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}

# (rows, dim, dtype): whole 16-byte vectors with 1 to 32 lanes per slot, two
# column blocks (dim 256 fp32), and element-wise rows (dims 3 and 1000 fp16)
MIXED = [(50, 4, "f32"), (70, 8, "f16"), (33, 12, "f32"), (40, 3, "f32"), (64, 64, "bf16"),
         (20, 256, "f32"), (16, 1000, "f16"), (300, 128, "f32"), (90, 32, "f16")]


def mixed_problem(seed, B, index_dtype, oob):
    rng = np.random.default_rng(seed)
    tables = []
    for rows, dim, dt in MIXED:
        w = torch.from_numpy(rng.standard_normal((rows, dim)).astype(np.float32))
        tables.append(w.to(TORCH_DT[dt]).to(DEV))
    T = len(MIXED)
    lengths = rng.integers(0, 21, size=T * B)
    lengths[::7] = 0
    idx = []
    for t, (rows, _, _) in enumerate(MIXED):
        n = int(lengths[t * B:(t + 1) * B].sum())
        ii = rng.integers(0, rows, size=n)
        if oob and n:
            k = rng.integers(0, n, size=max(1, n // 10))
            ii[k] = rng.choice([-1, rows, rows + 5], size=k.size)
        idx.append(ii)
    ind = np.concatenate(idx).astype(np.int64)
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    G = rng.standard_normal((B, sum(d for _, d, _ in MIXED))).astype(np.float32)
    tdt = torch.int64 if index_dtype == "i64" else torch.int32
    return tables, ind, off, G, tdt


def allowance(W, ind, off, B, G, pooling):
    """Per lookup: the rounding allowance of its D-term dot product.  W: the
    tables' values (float64 arrays)."""
    N = ind.shape[0]
    abs_dot = np.zeros(N)
    dims = np.ones(N)
    scale = np.ones(N)
    doff = 0
    for t, Wt in enumerate(W):
        R, D = Wt.shape
        lens = np.diff(off[t * B:(t + 1) * B + 1])
        s, e = off[t * B], off[(t + 1) * B]
        bag = np.repeat(np.arange(B), lens)
        r = ind[s:e]
        ok = (r >= 0) & (r < R)
        rr = np.where(ok, r, 0)
        d = np.abs(G[bag, doff:doff + D].astype(np.float64) * Wt[rr]).sum(1)
        abs_dot[s:e] = np.where(ok, d, 0.0)
        dims[s:e] = D
        if pooling == "mean":
            scale[s:e] = 1.0 / np.maximum(np.repeat(lens, lens), 1)
        doff += D
    return accumulation_allowance(abs_dot, dims, scale)


def values(tables):
    return [oracle.decode(DT_NAME[t.dtype], table_bits(t)) for t in tables]


@pytest.mark.parametrize("pooling", ["sum", "mean"])
@pytest.mark.parametrize("index_dtype", ["i64", "i32"])
@pytest.mark.parametrize("oob", [False, True])
def test_wgrad_mixed_tables(pooling, index_dtype, oob):
    B = 37
    tables, ind, off, G, tdt = mixed_problem(5 + int(oob), B, index_dtype, oob)
    h = tbe.tbe_create(tables, pooling)
    got = tbe.tbe_per_sample_weight_grad(h, torch.from_numpy(ind).to(tdt).to(DEV),
                                         torch.from_numpy(off).to(tdt).to(DEV), B,
                                         torch.from_numpy(G).to(DEV)).cpu().numpy()
    err = tbe.tbe_get_error(h)
    assert err == (tbe.TBE_ERR_INDEX_OOB if oob else tbe.TBE_OK)
    ref = oracle.weight_grad([table_bits(t) for t in tables], [DT_NAME[t.dtype] for t in tables], ind, off, B, G,
                             pooling=pooling)
    tol = dict(FP32_TOL)
    tol["atol"] = tol["atol"] + allowance(values(tables), ind, off, B, G, pooling)
    assert_close(got, ref, what=f"wgrad {pooling} {index_dtype}", **tol)
    if oob:
        bad = np.zeros(ind.shape[0], bool)
        for t, tab in enumerate(tables):
            s, e = off[t * B], off[(t + 1) * B]
            bad[s:e] = (ind[s:e] < 0) | (ind[s:e] >= tab.shape[0])
        assert bad.any() and not got[bad].any()
    h.close()


@pytest.mark.parametrize("cid", [1, 2, 3, 4, 5])
def test_wgrad_scaled_workloads(cid):
    cfg, tables, batch, grad = make_problem(cid)
    h = tbe.tbe_create(tables, cfg.pooling)
    got = tbe.tbe_per_sample_weight_grad(h, batch.indices.to(DEV), batch.offsets.to(DEV), cfg.B,
                                         grad.to(DEV)).cpu().numpy()
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    ind, off, G = batch.indices.numpy(), batch.offsets.numpy(), grad.numpy()
    ref = oracle.weight_grad([table_bits(t) for t in tables], [DT_NAME[t.dtype] for t in tables], ind, off, cfg.B,
                             G, pooling=cfg.pooling)
    tol = dict(FP32_TOL)
    tol["atol"] = tol["atol"] + allowance(values(tables), ind, off, cfg.B, G, cfg.pooling)
    assert_close(got, ref, what=f"cfg{cid} wgrad", **tol)
    h.close()


def test_wgrad_full_size_workload_3():
    """T=32 mixed bf16/fp16 tables, mean pooling, weighted, B=16384: sampled
    bags against the oracle on compact inputs, and at full size the identity
    sum_i w_i dL/dw_i = sum(out * G) (the forward pass is linear in w)."""
    cfg = workloads.get_config(3)
    specs = workloads.realize_tables(cfg)
    T, B = len(specs), cfg.B
    tables = workloads.make_tables(cfg, DEV, specs)
    batch = workloads.make_batch(cfg, DEV, torch.int64, specs)
    grad = workloads.make_grad(cfg, DEV, specs)
    h = tbe.tbe_create(tables, cfg.pooling)
    out = tbe.tbe_forward(h, batch.indices, batch.offsets, B, batch.weights)
    gw = tbe.tbe_per_sample_weight_grad(h, batch.indices, batch.offsets, B, grad)
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    lhs = torch.dot(batch.weights.double(), gw.double()).item()
    rhs = (out.double() * grad.double()).sum().item()
    scale = torch.dot(batch.weights.double(), gw.double().abs()).item()
    assert abs(lhs - rhs) <= 1e-5 * scale, (lhs, rhs, scale)

    # sampled bags: each with the rows it looks up, as a compact problem
    ind, off = batch.indices.cpu().numpy(), batch.offsets.cpu().numpy()
    rng = np.random.default_rng(303)
    bsample = np.sort(rng.choice(B, size=40, replace=False))
    c_tabs, c_dt, c_ind, c_len, pos_all = [], [], [], [], []
    for t in range(T):
        sl = [np.arange(off[t * B + b], off[t * B + b + 1]) for b in bsample]
        pos = np.concatenate(sl)
        uniq_rows, remap = np.unique(ind[pos], return_inverse=True)
        rows_t = uniq_rows if len(uniq_rows) else np.array([0])
        c_tabs.append(table_bits(tables[t][torch.from_numpy(rows_t).to(DEV)].cpu()))
        c_dt.append(DT_NAME[tables[t].dtype])
        c_ind.append(remap)
        c_len += [len(x) for x in sl]
        pos_all.append(pos)
    c_off = np.concatenate([[0], np.cumsum(c_len)]).astype(np.int64)
    c_G = grad[torch.from_numpy(bsample).to(DEV)].cpu().numpy()
    ref = oracle.weight_grad(c_tabs, c_dt, np.concatenate(c_ind).astype(np.int64), c_off, len(bsample), c_G,
                             pooling=cfg.pooling)
    got = gw.cpu().numpy()[np.concatenate(pos_all)]
    c_W = [oracle.decode(dt, tb) for tb, dt in zip(c_tabs, c_dt)]
    tol = dict(FP32_TOL)
    tol["atol"] = tol["atol"] + allowance(c_W, np.concatenate(c_ind), c_off, len(bsample), c_G, cfg.pooling)
    assert_close(got, ref, what="cfg3 sampled wgrad", **tol)
    h.close()


def test_wgrad_empty_and_bad_offsets():
    tables = [torch.randn(10, 8, device=DEV), torch.randn(5, 4, device=DEV)]
    h = tbe.tbe_create(tables, "sum")
    B = 3
    # every bag empty
    off = torch.zeros(2 * B + 1, dtype=torch.int64, device=DEV)
    ind = torch.zeros(0, dtype=torch.int64, device=DEV)
    g = torch.randn(B, 12, device=DEV)
    out = tbe.tbe_per_sample_weight_grad(h, ind, off, B, g)
    assert out.numel() == 0 and tbe.tbe_get_error(h) == tbe.TBE_OK
    # offsets that do not end at N
    ind = torch.tensor([1, 2, 3, 0], dtype=torch.int64, device=DEV)
    off = torch.tensor([0, 1, 2, 2, 3, 3, 3], dtype=torch.int64, device=DEV)
    tbe.tbe_per_sample_weight_grad(h, ind, off, B, g)
    assert tbe.tbe_get_error(h) == tbe.TBE_ERR_BAD_OFFSETS
    # null gradient pointer
    with pytest.raises(tbe.TBEError):
        tbe.tbe_per_sample_weight_grad(h, ind, off, B, None)
    h.close()
