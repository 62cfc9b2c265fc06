"""Pins for the CPU oracle: each function is checked against something other
than itself (hand-worked cases from the pages, library routines in float64,
a dense matrix formulation, closed forms and invariants)."""

import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *rest = line.split()
            vals.setdefault(k, []).append([float(x) for x in rest])
    return vals


# ----------------------------------------------------------------- problems

def random_problem(seed, T=3, B=7, dims=(4, 8, 12), rows=(9, 17, 5), dtypes=("f32", "f16", "bf16"),
                   max_len=6, index_dtype=np.int64, weights=False, oob=False):
    """Small random multi-table CSR problem with ragged and empty bags."""
    rng = np.random.default_rng(seed)
    tables_t = []
    for t in range(T):
        w = torch.from_numpy(rng.standard_normal((rows[t], dims[t]))).to(torch.float32)
        tables_t.append(w.to(TORCH_DT[dtypes[t]]))
    lengths = rng.integers(0, max_len + 1, size=T * B)
    lengths[::5] = 0  # some empty bags
    idx = []
    for t in range(T):
        n = int(lengths[t * B:(t + 1) * B].sum())
        ii = rng.integers(0, rows[t], size=n)
        if oob and n:
            k = rng.integers(0, n, size=max(1, n // 6))
            ii[k] = rng.choice([-1, rows[t], rows[t] + 3], size=k.size)
        idx.append(ii)
    indices = np.concatenate(idx).astype(index_dtype)
    offsets = np.concatenate([[0], np.cumsum(lengths)]).astype(index_dtype)
    w = rng.random(indices.shape[0]).astype(np.float32) if weights else None
    return tables_t, list(dtypes), indices, offsets, w, lengths


def np_tables(tables_t):
    """torch tables -> oracle arrays (float32, or uint16 bit patterns)."""
    out = []
    for w in tables_t:
        if w.dtype == torch.float32:
            out.append(w.numpy().copy())
        else:
            out.append(w.view(torch.int16).numpy().view(np.uint16).copy())
    return out


def torch_reference_forward(tables_t, indices, offsets, B, weights, pooling):
    """Per table, torch CPU embedding_bag in float64; concatenated on columns.
    Out-of-range lookups are routed to an appended zero row."""
    T = len(tables_t)
    cols = []
    for t, w in enumerate(tables_t):
        R = w.shape[0]
        w64 = torch.cat([w.to(torch.float64), torch.zeros(1, w.shape[1], dtype=torch.float64)])
        o = offsets[t * B:(t + 1) * B + 1].astype(np.int64)
        ii = indices[o[0]:o[-1]].astype(np.int64)
        ii = np.where((ii < 0) | (ii >= R), R, ii)
        lens = np.diff(o)
        psw = None
        if weights is not None:
            psw = torch.from_numpy(weights[o[0]:o[-1]].astype(np.float64))
        mode = pooling
        if pooling == "mean" and psw is not None:
            # mean with weights: sum of w_i x_i divided by the bag length
            psw = psw / torch.from_numpy(np.repeat(lens, lens).astype(np.float64))
            mode = "sum"
        r = F.embedding_bag(torch.from_numpy(ii), w64, torch.from_numpy(o - o[0]),
                            mode=mode, per_sample_weights=psw, include_last_offset=True)
        cols.append(r)
    return torch.cat(cols, 1).to(torch.float32).numpy()


# ------------------------------------------------------------ forward pins

def test_forward_worked_call_from_integration_page():
    g = read_golden("p1_call_example.txt")
    R, D = int(g["rows"][0][0]), int(g["dim"][0][0])
    W = np.repeat(np.arange(R, dtype=np.float32)[:, None], D, 1)
    indices = np.array(g["indices"][0], dtype=np.int64)
    offsets = np.array(g["offsets"][0], dtype=np.int64)
    out, skipped = oracle.forward([W], ["f32"], indices, offsets, B=2)
    assert skipped == 0
    np.testing.assert_array_equal(out, np.array(g["expected"], dtype=np.float32))


@pytest.mark.parametrize("pooling", ["sum", "mean"])
@pytest.mark.parametrize("weights", [False, True])
@pytest.mark.parametrize("index_dtype", [np.int32, np.int64])
def test_forward_matches_torch_embedding_bag(pooling, weights, index_dtype):
    for seed in range(4):
        tabs, dts, ind, off, w, _ = random_problem(seed, index_dtype=index_dtype, weights=weights)
        out, skipped = oracle.forward(np_tables(tabs), dts, ind, off, B=7, weights=w,
                                      pooling=pooling)
        assert skipped == 0
        ref = torch_reference_forward(tabs, ind, off, 7, w, pooling)
        np.testing.assert_array_max_ulp(out, ref, maxulp=1)


def test_forward_dense_matrix_formulation():
    """out_t = A_t @ W_t with A_t[b, r] = sum of s_i over the bag's lookups of r."""
    tabs, dts, ind, off, w, lengths = random_problem(11, weights=True, max_len=9)
    B = 7
    out, _ = oracle.forward(np_tables(tabs), dts, ind, off, B=B, weights=w)
    col = 0
    for t, wt in enumerate(tabs):
        R, D = wt.shape
        A = np.zeros((B, R))
        for b in range(B):
            lo, hi = off[t * B + b], off[t * B + b + 1]
            np.add.at(A[b], ind[lo:hi].astype(np.int64), w[lo:hi].astype(np.float64))
        ref = A @ wt.to(torch.float64).numpy()
        np.testing.assert_allclose(out[:, col:col + D], ref, rtol=2e-7, atol=1e-12)
        col += D


def test_forward_out_of_range_lookups_are_skipped():
    tabs, dts, ind, off, w, _ = random_problem(5, weights=True, oob=True, max_len=8)
    for pooling in ("sum", "mean"):
        out, skipped = oracle.forward(np_tables(tabs), dts, ind, off, B=7, weights=w,
                                      pooling=pooling)
        rows = [t.shape[0] for t in tabs]
        bag_table = np.repeat(np.arange(3), 7)
        lens = np.diff(off)
        tab_of = np.repeat(bag_table, lens)
        expect_skipped = int(sum(((ind[tab_of == t] < 0) | (ind[tab_of == t] >= rows[t])).sum()
                                 for t in range(3)))
        assert skipped == expect_skipped > 0
        ref = torch_reference_forward(tabs, ind, off, 7, w, pooling)
        np.testing.assert_array_max_ulp(out, ref, maxulp=1)


def test_forward_rejects_bad_offsets():
    W = np.zeros((4, 2), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.forward([W], ["f32"], np.array([0, 1, 2]), np.array([0, 2, 1, 3]), B=3)
    with pytest.raises(oracle.OracleError):
        oracle.forward([W], ["f32"], np.array([0, 1, 2]), np.array([0, 1, 2]), B=2)


# ---------------------------------------------------- storage conversions

def test_decode_every_f16_and_bf16_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode("f16", bits)
    ref = bits.view(np.float16).astype(np.float64)
    np.testing.assert_array_equal(got, ref)  # NaNs compare equal in assert_array_equal
    got = oracle.decode("bf16", bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(got, ref)


def test_round_f16_matches_numpy():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 5, 20000),
        rng.uniform(-70000, 70000, 2000),
        [0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6, 2.0 ** -24, 2.0 ** -25,
         3 * 2.0 ** -26, 2.0 ** -14, np.inf, -np.inf],
    ])
    # exact midpoints between adjacent binary16 values (ties go to even)
    h = np.arange(0, 0x7bff, 7, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (h[:-1] + np.nextafter(h[:-1].astype(np.float16), np.float16(np.inf)).astype(
        np.float64)) / 2
    x = np.concatenate([x, mids, -mids])
    got = oracle.round_to("f16", x)
    ref = x.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_round_bf16_single_rounding():
    rng = np.random.default_rng(1)
    # values exactly representable in fp32: torch's fp32 -> bf16 is then a single rounding
    x32 = (rng.standard_normal(50000) * 10.0 ** rng.integers(-30, 30, 50000)).astype(np.float32)
    x32 = np.concatenate([x32, np.float32([0.0, -0.0, 3.3895314e38, 1e-40, -1e-45, np.inf])])
    got = oracle.round_to("bf16", x32.astype(np.float64))
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, ref)
    # exact ties between neighbours: the neighbour with an even last bit wins
    lo = np.arange(0x3f00, 0x4100, dtype=np.uint16)
    lo_v = oracle.decode("bf16", lo)
    hi_v = oracle.decode("bf16", lo + 1)
    got = oracle.round_to("bf16", (lo_v + hi_v) / 2)
    expect = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint16)
    np.testing.assert_array_equal(got, expect)


# ------------------------------------------------- transpose, sort and RLE

def test_make_keys_bag_assignment():
    tabs, dts, ind, off, _, lengths = random_problem(3, oob=True, max_len=7)
    rows = [t.shape[0] for t in tabs]
    keys, bag = oracle.make_keys(rows, ind, off, B=7)
    np.testing.assert_array_equal(bag, np.repeat(np.arange(21), lengths))
    t_of = bag // 7
    rowbase = np.concatenate([[0], np.cumsum(rows)])
    valid = (ind >= 0) & (ind < np.array(rows)[t_of])
    np.testing.assert_array_equal(keys[valid], rowbase[t_of[valid]] + ind[valid])
    assert (keys[~valid] == sum(rows)).all() and (~valid).any()


@pytest.mark.parametrize("n,hi", [(0, 5), (1, 5), (1000, 7), (5000, 300), (20000, 1 << 27)])
def test_sort_rle_matches_numpy(n, hi):
    rng = np.random.default_rng(n + hi)
    keys = rng.integers(0, hi, size=n)
    r = oracle.sort_rle(keys)
    perm = np.argsort(keys, kind="stable")
    np.testing.assert_array_equal(r["sorted_pos"], perm)
    np.testing.assert_array_equal(r["sorted_keys"], keys[perm])
    u, first, counts = np.unique(keys[perm], return_index=True, return_counts=True)
    np.testing.assert_array_equal(r["uniq"], u)
    np.testing.assert_array_equal(r["runstart"], first)
    np.testing.assert_array_equal(r["runlen"], counts)


# ------------------------------------------------------------ backward pins

def torch_grads(tabs, ind, off, B, w, pooling, G):
    """W.grad of sum(out * G) through torch CPU embedding_bag in float64."""
    leaves = [t.to(torch.float64).requires_grad_(True) for t in tabs]
    outs = []
    for t, wt in enumerate(leaves):
        o = off[t * B:(t + 1) * B + 1].astype(np.int64)
        ii = torch.from_numpy(ind[o[0]:o[-1]].astype(np.int64))
        psw = None if w is None else torch.from_numpy(w[o[0]:o[-1]].astype(np.float64))
        mode = pooling
        if pooling == "mean" and psw is not None:
            lens = np.diff(o)
            psw = psw / torch.from_numpy(np.repeat(lens, lens).astype(np.float64))
            mode = "sum"
        outs.append(F.embedding_bag(ii, wt, torch.from_numpy(o - o[0]), mode=mode,
                                    per_sample_weights=psw, include_last_offset=True))
    out = torch.cat(outs, 1)
    (out * torch.from_numpy(G.astype(np.float64))).sum().backward()
    return [l.grad.numpy() for l in leaves]


@pytest.mark.parametrize("pooling", ["sum", "mean"])
@pytest.mark.parametrize("weights", [False, True])
def test_row_grads_match_torch_autograd(pooling, weights):
    for seed in range(3):
        tabs, dts, ind, off, w, _ = random_problem(20 + seed, weights=weights, max_len=8)
        B = 7
        G = np.random.default_rng(seed).standard_normal((B, 24)).astype(np.float32)
        tabs_np = np_tables(tabs)
        rk, rg = oracle.backward(tabs_np, dts, ind, off, B, G, "none", 0.0, weights=w,
                                 pooling=pooling, want_row_grads=True)
        ref = torch_grads(tabs, ind, off, B, w, pooling, G)
        rows = [t.shape[0] for t in tabs]
        rowbase = np.concatenate([[0], np.cumsum(rows)])
        seen = [np.zeros(r, bool) for r in rows]
        for k, g in zip(rk, rg):
            t = int(np.searchsorted(rowbase, k, side="right") - 1)
            r = int(k - rowbase[t])
            D = tabs[t].shape[1]
            np.testing.assert_allclose(g[:D], ref[t][r], rtol=1e-12, atol=1e-12)
            seen[t][r] = True
        for t in range(3):  # rows never looked up have zero gradient
            assert not ref[t][~seen[t]].any()


def test_row_grad_column_sum_invariant():
    """sum over rows of g_t equals sum over bags of (sum of s_i) * G[bag, cols of t]."""
    tabs, dts, ind, off, w, lengths = random_problem(33, weights=True, max_len=9)
    B = 7
    G = np.random.default_rng(9).standard_normal((B, 24)).astype(np.float32)
    rk, rg = oracle.backward(np_tables(tabs), dts, ind, off, B, G, "none", 0.0, weights=w,
                             want_row_grads=True)
    rows = [t.shape[0] for t in tabs]
    rowbase = np.concatenate([[0], np.cumsum(rows)])
    t_of_key = np.searchsorted(rowbase, rk, side="right") - 1
    col = 0
    for t in range(3):
        D = tabs[t].shape[1]
        lhs = rg[t_of_key == t, :D].sum(0)
        ssum = np.array([w[off[t * B + b]:off[t * B + b + 1]].astype(np.float64).sum()
                         for b in range(B)])
        rhs = ssum @ G[:, col:col + D].astype(np.float64)
        np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)
        col += D


def test_repeated_row_hand_case():
    g = read_golden("repeated_row_backward.txt")
    R, D = int(g["rows"][0][0]), int(g["dim"][0][0])
    W = np.zeros((R, D), np.float32)
    W[3] = g["w3"][0]
    ind = np.array(g["indices"][0], np.int64)
    off = np.array(g["offsets"][0], np.int64)
    G = np.array([g["grad"][0]], np.float32)
    lr = g["lr"][0][0]
    rk, rg = oracle.backward([W], ["f32"], ind, off, 1, G, "sgd", lr, want_row_grads=True)
    assert list(rk) == [3]
    np.testing.assert_array_equal(rg[0], g["expected_grad"][0])
    np.testing.assert_array_equal(W[3], np.array(g["expected_w3"][0], np.float32))
    assert not W[[0, 1, 2, 4]].any()


def test_sgd_matches_torch_optim_and_touches_only_looked_up_rows():
    tabs, dts, ind, off, w, _ = random_problem(41, dtypes=("f32", "f32", "f32"), weights=True,
                                               max_len=8)
    B = 7
    lr = float(np.float32(0.01))
    G = np.random.default_rng(2).standard_normal((B, 24)).astype(np.float32)
    before = np_tables(tabs)
    after = [t.copy() for t in before]
    oracle.backward(after, dts, ind, off, B, G, "sgd", lr, weights=w)
    grads = torch_grads(tabs, ind, off, B, w, "sum", G)
    for t in range(3):
        p = torch.from_numpy(before[t].astype(np.float64)).requires_grad_(True)
        p.grad = torch.from_numpy(grads[t])
        torch.optim.SGD([p], lr=lr).step()
        np.testing.assert_array_max_ulp(after[t], p.detach().numpy().astype(np.float32), maxulp=1)
        touched = np.unique(ind[np.repeat(np.arange(21) // 7, np.diff(off)) == t])
        untouched = np.setdiff1d(np.arange(before[t].shape[0]), touched)
        np.testing.assert_array_equal(after[t][untouched], before[t][untouched])
        assert (after[t][touched] != before[t][touched]).any(axis=1).all()


def test_rowwise_adagrad_dim1_is_torch_adagrad():
    """With one column, mean_j g_j^2 = g^2: row-wise Adagrad is torch.optim.Adagrad."""
    rng = np.random.default_rng(5)
    R, B = 13, 6
    W = rng.standard_normal((R, 1)).astype(np.float32)
    lr, eps = float(np.float32(0.05)), float(np.float32(1e-3))
    state = np.zeros(R, np.float32)
    ours = W.copy()
    p = torch.from_numpy(W.astype(np.float64)).requires_grad_(True)
    opt = torch.optim.Adagrad([p], lr=lr, eps=eps, initial_accumulator_value=0.0)
    for step in range(3):
        lens = rng.integers(0, 5, B)
        ind = rng.integers(0, R, int(lens.sum()))
        off = np.concatenate([[0], np.cumsum(lens)])
        G = rng.standard_normal((B, 1)).astype(np.float32)
        oracle.backward([ours], ["f32"], ind, off, B, G, "adagrad", lr, eps=eps, state=state)
        opt.zero_grad()
        out = F.embedding_bag(torch.from_numpy(ind), p, torch.from_numpy(off),
                              mode="sum", include_last_offset=True)
        (out * torch.from_numpy(G.astype(np.float64))).sum().backward()
        opt.step()
        np.testing.assert_allclose(ours[:, 0], p.detach().numpy()[:, 0], rtol=2e-7, atol=1e-9)
        np.testing.assert_allclose(state, opt.state[p]["sum"].numpy()[:, 0], rtol=2e-7, atol=0)


def test_rowwise_adagrad_equal_magnitude_rows_is_torch_adagrad():
    """If every column of a row's gradient has the same magnitude, the row-wise
    state mean_j g_j^2 equals each column's element-wise Adagrad state."""
    rng = np.random.default_rng(6)
    R, D, B = 11, 4, 9
    W = rng.standard_normal((R, D)).astype(np.float32)
    lr, eps = float(np.float32(0.1)), float(np.float32(1e-6))
    sign = np.array([1, -1, -1, 1], np.float64)
    lens = rng.integers(1, 5, B)
    ind = rng.integers(0, R, int(lens.sum()))
    off = np.concatenate([[0], np.cumsum(lens)])
    c = rng.uniform(0.5, 2.0, B)
    G = (c[:, None] * sign[None, :]).astype(np.float32)
    state = np.zeros(R, np.float32)
    ours = W.copy()
    oracle.backward([ours], ["f32"], ind, off, B, G, "adagrad", lr, eps=eps, state=state)
    p = torch.from_numpy(W.astype(np.float64)).requires_grad_(True)
    opt = torch.optim.Adagrad([p], lr=lr, eps=eps, initial_accumulator_value=0.0)
    out = F.embedding_bag(torch.from_numpy(ind), p, torch.from_numpy(off), mode="sum",
                          include_last_offset=True)
    (out * torch.from_numpy(G.astype(np.float64))).sum().backward()
    opt.step()
    np.testing.assert_allclose(ours, p.detach().numpy(), rtol=2e-7, atol=1e-9)
    np.testing.assert_allclose(state, opt.state[p]["sum"].numpy()[:, 0], rtol=2e-7, atol=0)


def test_rowwise_adagrad_closed_form():
    g = read_golden("rowwise_adagrad_closed_form.txt")
    R, D = int(g["rows"][0][0]), int(g["dim"][0][0])
    c, lr = g["c"][0][0], g["lr"][0][0]
    W = np.full((R, D), g["w0"][0][0], np.float32)
    state = np.zeros(R, np.float32)
    ind, off = np.array([1], np.int64), np.array([0, 1], np.int64)
    G = np.full((1, D), c, np.float32)
    for step in range(2):
        oracle.backward([W], ["f32"], ind, off, 1, G, "adagrad", lr, eps=0.0, state=state)
        assert state[1] == np.float32(g["expected_m"][0][step])
        np.testing.assert_array_max_ulp(W[1], np.full(D, g["expected_w"][0][step], np.float32),
                                        maxulp=1)
        assert state[0] == 0 and (W[0] == g["w0"][0][0]).all()


def test_backward_low_precision_rows_round_once():
    """fp16/bf16 rows: the update is computed in double and rounded once."""
    tabs, dts, ind, off, w, _ = random_problem(50, weights=True, max_len=6)
    B = 7
    G = np.random.default_rng(4).standard_normal((B, 24)).astype(np.float32)
    lr = float(np.float32(0.25))
    before = np_tables(tabs)
    after = [t.copy() for t in before]
    oracle.backward(after, dts, ind, off, B, G, "sgd", lr, weights=w)
    grads = torch_grads(tabs, ind, off, B, w, "sum", G)
    for t in range(3):
        exact = oracle.decode(dts[t], before[t]) - lr * grads[t]
        expect = oracle.round_to(dts[t], exact)
        if dts[t] == "f16":
            np.testing.assert_array_equal(after[t], exact.astype(np.float16).view(np.uint16))
        np.testing.assert_array_equal(after[t], expect)


# ------------------------------------------------- per-sample weight gradient

def torch_weight_grad(tabs, ind, off, B, w, pooling, G):
    """per_sample_weights.grad of sum(out * G) through torch CPU embedding_bag in
    float64; out-of-range lookups are routed to an appended zero row."""
    leaf = torch.from_numpy(w.astype(np.float64)).requires_grad_(True)
    outs = []
    for t, wt in enumerate(tabs):
        R = wt.shape[0]
        w64 = torch.cat([wt.to(torch.float64), torch.zeros(1, wt.shape[1], dtype=torch.float64)])
        o = off[t * B:(t + 1) * B + 1].astype(np.int64)
        ii = ind[o[0]:o[-1]].astype(np.int64)
        ii = np.where((ii < 0) | (ii >= R), R, ii)
        psw = leaf[o[0]:o[-1]]
        if pooling == "mean":
            lens = np.diff(o)
            psw = psw / torch.from_numpy(np.repeat(lens, lens).astype(np.float64))
        outs.append(F.embedding_bag(torch.from_numpy(ii), w64, torch.from_numpy(o - o[0]), mode="sum",
                                    per_sample_weights=psw, include_last_offset=True))
    (torch.cat(outs, 1) * torch.from_numpy(G.astype(np.float64))).sum().backward()
    return leaf.grad.numpy()


@pytest.mark.parametrize("pooling", ["sum", "mean"])
@pytest.mark.parametrize("oob", [False, True])
def test_weight_grad_matches_torch_autograd(pooling, oob):
    for seed in range(3):
        tabs, dts, ind, off, w, _ = random_problem(40 + seed, weights=True, max_len=8, oob=oob)
        B = 7
        G = np.random.default_rng(seed).standard_normal((B, 24)).astype(np.float32)
        got = oracle.weight_grad(np_tables(tabs), dts, ind, off, B, G, pooling=pooling)
        ref = torch_weight_grad(tabs, ind, off, B, w, pooling, G)
        np.testing.assert_allclose(got, ref.astype(np.float32), rtol=1e-6, atol=1e-7)
        if oob:
            rows = [t.shape[0] for t in tabs]
            for t in range(3):
                lo, hi = off[t * B], off[(t + 1) * B]
                bad = (ind[lo:hi] < 0) | (ind[lo:hi] >= rows[t])
                assert not got[lo:hi][bad].any()


def test_weight_grad_euler_identity():
    """out is linear in the weights, so sum_i w_i dL/dw_i = sum(out * G)."""
    tabs, dts, ind, off, w, _ = random_problem(51, weights=True, max_len=9)
    B = 7
    G = np.random.default_rng(4).standard_normal((B, 24)).astype(np.float32)
    for pooling in ("sum", "mean"):
        out, _ = oracle.forward(np_tables(tabs), dts, ind, off, B, weights=w, pooling=pooling)
        gw = oracle.weight_grad(np_tables(tabs), dts, ind, off, B, G, pooling=pooling)
        lhs = float(np.dot(w.astype(np.float64), gw.astype(np.float64)))
        rhs = float((out.astype(np.float64) * G.astype(np.float64)).sum())
        assert lhs == pytest.approx(rhs, rel=1e-5, abs=1e-6)


def test_weight_grad_hand_case():
    """One table of two rows, D = 2; bag 0 = rows (1, 0, 1), bag 1 empty."""
    W = np.array([[1.0, 2.0], [3.0, -1.0]], np.float32)
    ind = np.array([1, 0, 1], np.int64)
    off = np.array([0, 3, 3], np.int64)
    G = np.array([[0.5, 2.0], [7.0, 7.0]], np.float32)
    got = oracle.weight_grad([W], ["f32"], ind, off, 2, G)
    # row 1 . G[0] = 1.5 - 2 = -0.5; row 0 . G[0] = 0.5 + 4 = 4.5
    np.testing.assert_array_equal(got, np.array([-0.5, 4.5, -0.5], np.float32))
    got = oracle.weight_grad([W], ["f32"], ind, off, 2, G, pooling="mean")
    np.testing.assert_allclose(got, np.array([-0.5, 4.5, -0.5], np.float32) / 3, rtol=1e-7)


# ------------------------------------------- timing build (CPU baseline)

@pytest.mark.parametrize("optimizer", ["sgd", "adagrad"])
def test_timing_build_gives_the_plain_builds_results(optimizer):
    """bench.py times the oracle's OpenMP build on all host cores; each bag's
    and each run's sums are the same additions in the same order, so its
    outputs, updated rows and state are bit-identical to the pinned build."""
    tabs, dts, ind, off, w, _ = random_problem(51, dtypes=("f32", "f16", "bf16"), weights=True, max_len=40,
                                               oob=True)
    B = 7
    G = np.random.default_rng(3).standard_normal((B, 24)).astype(np.float32)
    results = []
    try:
        for build in ("plain", "timing"):
            if build == "timing":
                assert oracle.use_timing_build(4) >= 1
            out, skipped = oracle.forward(np_tables(tabs), dts, ind, off, B, weights=w, pooling="mean")
            after = np_tables(tabs)
            state = np.zeros(sum(t.shape[0] for t in tabs), np.float32)
            oracle.backward(after, dts, ind, off, B, G, optimizer, 0.05, eps=1e-8, weights=w, pooling="mean",
                            state=state)
            results.append((out, skipped, after, state))
    finally:
        oracle.use_plain_build()
    (o0, s0, a0, st0), (o1, s1, a1, st1) = results
    assert s0 == s1 and s0 > 0
    np.testing.assert_array_equal(o0.view(np.uint32), o1.view(np.uint32))
    for x, y in zip(a0, a1):
        np.testing.assert_array_equal(x.view(np.uint8), y.view(np.uint8))
    np.testing.assert_array_equal(st0.view(np.uint32), st1.view(np.uint32))
