"""GPU parity at the workloads' full sizes, in the configuration bench.py
times (default handle flags, int64 indices: small tables take the dense
backward and stay out of the sort).

Full tables (4 to 20 GB) are too large for the oracle, so the checks are:
  - sort and run-length encoding: the whole sorted key array, sorted
    positions, distinct keys and run starts, bit-exact against numpy's stable
    argsort of the keys the oracle's transpose step produces;
  - forward: sampled bags, recomputed by the oracle on compact inputs (each
    sampled bag with the rows it looks up);
  - backward: sampled rows (the hottest rows, random looked-up rows, rows
    nobody looks up).  For a sampled row, every lookup that hits it becomes a
    one-lookup bag of the compact problem with the lookup's scale s_i as its
    weight and its bag's upstream gradient row, so the oracle's per-row sum
    and optimizer step see exactly the lookups the full batch has; rows no
    lookup touches must come back bit-identical.
"""

import numpy as np
import pytest
import torch

import oracle
import recommender_sparse_embeddings_gb300 as tbe
import workloads
from helpers import (DT_NAME, FP32_TOL, LOWP_TOL, accumulation_allowance, assert_close, histogram_allowance,
                     table_bits)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _rows_host(t: torch.Tensor, rows: np.ndarray) -> torch.Tensor:
    return t[torch.from_numpy(rows).to(t.device)].cpu()


@pytest.mark.parametrize("cid", [2, 3, 4, 5])
def test_full_size(cid):
    cfg = workloads.get_config(cid)
    specs = workloads.realize_tables(cfg)
    T, B = len(specs), cfg.B
    tables = workloads.make_tables(cfg, DEV, specs)
    batch = workloads.make_batch(cfg, DEV, torch.int64, specs)
    grad = workloads.make_grad(cfg, DEV, specs)
    N = batch.N
    rows = np.array([s.rows for s in specs], dtype=np.int64)
    dims = [s.dim for s in specs]
    doff = np.concatenate([[0], np.cumsum(dims)])
    ind = batch.indices.cpu().numpy()
    off = batch.offsets.cpu().numpy()
    w = None if batch.weights is None else batch.weights.cpu().numpy()
    rng = np.random.default_rng(100 + cid)

    h = tbe.tbe_create(tables, cfg.pooling)
    paths = tbe.tbe_table_paths(h)
    ws = tbe.make_workspace(h, N, B)
    out = tbe.tbe_forward_prepare(h, batch.indices, batch.offsets, B, ws, batch.weights)
    assert tbe.tbe_get_error(h) == tbe.TBE_OK

    # ---- sort / run-length: whole arrays, bit-exact (histogram tables take
    # the dense backward: only the other tables' keys are sorted)
    keys, bag_of = oracle.make_keys(rows, ind, off, B)
    dense = np.array([p == "dense" for p in tbe.tbe_backward_paths(h)])
    keep = np.flatnonzero(~dense[bag_of // B])
    Ns = len(keep)
    perm = np.argsort(keys[keep], kind="stable")
    skeys = keys[keep][perm]
    lay = tbe.tbe_backward_workspace_layout(h, N, B)

    def u32(offset, n):
        return ws[offset:offset + 4 * n].view(torch.int32).cpu().numpy().view(np.uint32).astype(np.int64)

    np.testing.assert_array_equal(u32(lay.sorted_keys, Ns), skeys)
    scaled = w is not None or cfg.pooling == "mean"  # values: positions, else flat bags
    np.testing.assert_array_equal(u32(lay.sorted_vals, Ns), keep[perm] if scaled else bag_of[keep[perm]])
    U = int(u32(lay.num_unique, 1)[0])
    head = np.flatnonzero(np.r_[True, skeys[1:] != skeys[:-1]])
    assert U == len(head)
    np.testing.assert_array_equal(u32(lay.uniq, U), skeys[head])
    np.testing.assert_array_equal(u32(lay.runstart, U + 1), np.r_[head, Ns])

    # ---- forward: sampled bags
    bsample = np.sort(rng.choice(B, size=48, replace=False))
    c_tabs, c_dt, c_ind, c_len, c_w = [], [], [], [], []
    for t in range(T):
        sl = [np.arange(off[t * B + b], off[t * B + b + 1]) for b in bsample]
        pos = np.concatenate(sl)
        uniq_rows, remap = np.unique(ind[pos], return_inverse=True)
        c_tabs.append(table_bits(_rows_host(tables[t], uniq_rows)) if len(uniq_rows) else
                      table_bits(tables[t][:1].cpu()))
        c_dt.append(DT_NAME[tables[t].dtype])
        c_ind.append(remap)
        c_len += [len(x) for x in sl]
        if w is not None:
            c_w.append(w[pos])
    c_off = np.concatenate([[0], np.cumsum(c_len)]).astype(np.int64)
    c_ind_all = np.concatenate(c_ind).astype(np.int64)
    c_w_all = None if w is None else np.concatenate(c_w)
    ref, skipped = oracle.forward(c_tabs, c_dt, c_ind_all, c_off, len(bsample), weights=c_w_all,
                                  pooling=cfg.pooling)
    assert skipped == 0
    # the histogram path's allowance: the terms' magnitudes (the oracle on
    # |W| and |w|) and the bag lengths
    abs_tabs = [np.abs(tb) if dt == "f32" else tb & np.uint16(0x7fff) for dt, tb in zip(c_dt, c_tabs)]
    abs_ref, _ = oracle.forward(abs_tabs, c_dt, c_ind_all, c_off, len(bsample),
                                weights=None if c_w_all is None else np.abs(c_w_all), pooling=cfg.pooling)
    c_lens = np.diff(c_off).reshape(T, len(bsample))
    got = out[torch.from_numpy(bsample).to(DEV)].cpu().numpy()
    for t in range(T):
        cols = slice(doff[t], doff[t + 1])
        atol = FP32_TOL["atol"]
        if paths[t] == "histogram":
            atol = atol + histogram_allowance(abs_ref[:, cols], c_lens[t][:, None])
        assert_close(got[:, cols], ref[:, cols], what=f"cfg{cid} forward table {t}", rtol=FP32_TOL["rtol"],
                     atol=atol)

    # ---- backward: sampled rows
    t_of = bag_of // B
    samples = []  # (table, rows touched, rows untouched)
    for t in sorted(rng.choice(T, size=min(T, 4), replace=False).tolist()):
        mask = t_of == t
        tr, counts = np.unique(ind[mask], return_counts=True)
        hot = tr[np.argsort(-counts, kind="stable")[:2]]
        rand = rng.choice(tr, size=min(12, len(tr)), replace=False)
        touched = np.unique(np.r_[hot, rand])
        untouched = np.setdiff1d(rng.choice(rows[t], size=min(int(rows[t]), 64), replace=False), tr)[:8]
        samples.append((t, touched, untouched))
    before = {t: (table_bits(_rows_host(tables[t], tr)), table_bits(_rows_host(tables[t], un)))
              for t, tr, un in samples}
    total_rows = int(rows.sum())
    state = torch.zeros(total_rows, dtype=torch.float32, device=DEV) if cfg.optimizer == "adagrad" else None
    tbe.tbe_backward_apply(h, N, B, grad, ws, cfg.optimizer, cfg.lr, cfg.eps, state)
    assert tbe.tbe_get_error(h) == tbe.TBE_OK
    G = grad.cpu().numpy()
    L_of_bag = np.diff(off)
    rowbase = np.concatenate([[0], np.cumsum(rows)])
    for t, touched, untouched in samples:
        name = DT_NAME[tables[t].dtype]
        w_tr, w_un = before[t]
        after_tr = table_bits(_rows_host(tables[t], touched))
        after_un = table_bits(_rows_host(tables[t], untouched))
        np.testing.assert_array_equal(after_un, w_un, err_msg=f"cfg{cid} table {t}: untouched rows changed")
        # compact problem: one bag per lookup of a sampled row
        hit = np.flatnonzero((t_of == t) & np.isin(ind, touched))
        remap = np.searchsorted(touched, ind[hit])
        s = np.ones(len(hit)) if w is None else w[hit].astype(np.float64)
        if cfg.pooling == "mean":
            s = s / L_of_bag[bag_of[hit]]
        c_grad = G[bag_of[hit] - t * B][:, doff[t]:doff[t + 1]]
        c_tab = w_tr.copy()
        c_state = np.zeros(len(touched), np.float32) if state is not None else None
        oracle.backward([c_tab], [name], remap.astype(np.int64), np.arange(len(hit) + 1, dtype=np.int64),
                        len(hit), c_grad, cfg.optimizer, cfg.lr, eps=cfg.eps, weights=s.astype(np.float32),
                        pooling="sum", state=c_state)
        tol = dict(FP32_TOL if name == "f32" else LOWP_TOL)
        # rounding allowance of the fp32 row sums (rows hit thousands of times)
        abs_terms = np.zeros((len(touched), c_grad.shape[1]))
        np.add.at(abs_terms, remap, np.abs(s[:, None] * c_grad.astype(np.float64)))
        n_terms = np.bincount(remap, minlength=len(touched))[:, None]
        scale = cfg.lr if state is None else cfg.lr / (np.sqrt(c_state.astype(np.float64)) + cfg.eps)[:, None]
        tol["atol"] = tol["atol"] + accumulation_allowance(abs_terms, n_terms, scale)
        assert_close(oracle.decode(name, after_tr), oracle.decode(name, c_tab), what=f"cfg{cid} table {t} rows",
                     **tol)
        if state is not None:
            got_state = state[torch.from_numpy(rowbase[t] + touched).to(DEV)].cpu().numpy()
            assert_close(got_state, c_state, what=f"cfg{cid} table {t} state", **FP32_TOL)
    h.close()
    del tables, batch, grad, ws, out
    torch.cuda.empty_cache()
