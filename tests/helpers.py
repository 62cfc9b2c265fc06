"""Shared helpers of the GPU parity tests: conversions between torch tensors
and the oracle's arrays, oracle calls, and tolerance checks."""

from __future__ import annotations

import numpy as np
import torch

import oracle

DT_NAME = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}

# Tolerances: |got - ref| <= atol + rtol * |ref|.
FP32_TOL = dict(rtol=1e-5, atol=1e-6)      # fp32 pooled outputs, fp32 updated rows, state
LOWP_TOL = dict(rtol=1e-2, atol=1e-6)      # fp16/bf16 rows after one rounding to storage


def table_bits(t: torch.Tensor) -> np.ndarray:
    """Torch table -> oracle array (float32, or raw uint16 bit patterns)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy().copy()
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def decoded(t_or_bits, dtype_name: str = None) -> np.ndarray:
    """Exact float64 values of a torch table or of oracle bits."""
    if isinstance(t_or_bits, torch.Tensor):
        dtype_name = DT_NAME[t_or_bits.dtype]
        t_or_bits = table_bits(t_or_bits)
    return oracle.decode(dtype_name, t_or_bits)


def np_index(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def accumulation_allowance(terms_abs_sum, n_terms, scale) -> np.ndarray:
    """Absolute error allowance for an updated row w - scale * g, where g is an
    fp32 sum of n_terms terms whose magnitudes add up to terms_abs_sum.

    Each fp32 addition rounds to nearest with relative error at most 2^-24 of
    a partial sum bounded by terms_abs_sum; taking those errors as
    independent, the error of g has a standard deviation of about
    sqrt(n) * 2^-24 * terms_abs_sum, and four of those are allowed.  The
    update multiplies that error by `scale` (lr for SGD, lr / (sqrt(m) + eps)
    for row-wise Adagrad).  Where w and scale * g nearly cancel, the relative
    tolerance on the small result is tighter than the fp32 gradient itself
    can be; this term covers exactly that."""
    n = np.asarray(n_terms, dtype=np.float64)
    return 4.0 * np.sqrt(n) * 2.0 ** -24 * np.asarray(terms_abs_sum, np.float64) * np.asarray(scale, np.float64)


def pooled_abs_sum(tables, indices, offsets, B, weights=None, pooling="sum"):
    """Per output element, the sum of the magnitudes of its terms,
    sum_i |s_i| * |W[idx_i, j]| (the oracle run on |W| and |w|), and the
    length of each output row's bag (per table, broadcast over its columns)."""
    abs_tabs = [t.abs() for t in tables]
    absw = None if weights is None else weights.abs()
    a, _ = oracle_forward(abs_tabs, indices, offsets, B, absw, pooling)
    off = np.asarray(np_index(offsets), dtype=np.int64)
    lens = np.diff(off).reshape(len(tables), B)
    n = np.concatenate([np.repeat(lens[t][:, None], int(tables[t].shape[1]), axis=1) for t in range(len(tables))],
                       axis=1)
    return a, n


def histogram_allowance(abs_sum, n_terms) -> np.ndarray:
    """Absolute error allowance of a pooled output of the tensor-core
    histogram path beyond the fp32 tolerance.

    Each histogram entry reaches the tensor cores as two fp16 terms hi + lo
    (bag-wise scaled into fp16's range), so it carries a relative error of at
    most 2^-22 (one fp16 rounding of lo, which is at most 2^-11 of the entry);
    2^-21 * abs_sum covers that.  The products are then summed in fp32, which
    rounds like any fp32 sum of n terms: 4 * sqrt(n) * 2^-24 * abs_sum, as in
    accumulation_allowance.  The allowance matters only where the output
    cancels to far below its terms."""
    n = np.maximum(np.asarray(n_terms, dtype=np.float64), 1.0)
    a = np.asarray(abs_sum, dtype=np.float64)
    return 2.0 ** -21 * a + 4.0 * np.sqrt(n) * 2.0 ** -24 * a


def assert_close(got, ref, rtol, atol, what=""):
    """|got - ref| <= atol + rtol * |ref| element-wise (atol may be an array)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        k = np.flatnonzero(bad.ravel())[:5]
        atol_at = np.broadcast_to(np.asarray(atol, np.float64), ref.shape).ravel()[k]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outside tol (rtol={rtol}, atol={atol_at.tolist()}); "
            f"first at flat {k.tolist()}: got {got.ravel()[k].tolist()} ref {ref.ravel()[k].tolist()}; "
            f"max abs err {err.max():.3e}")


def oracle_forward(tables, indices, offsets, B, weights=None, pooling="sum"):
    out, skipped = oracle.forward([table_bits(t) for t in tables], [DT_NAME[t.dtype] for t in tables],
                                  np_index(indices), np_index(offsets), B,
                                  weights=None if weights is None else np_index(weights),
                                  pooling=pooling)
    return out, skipped


def oracle_backward(tables, indices, offsets, B, grad, optimizer, lr, eps=0.0, weights=None,
                    pooling="sum", state=None):
    """Returns (updated oracle tables as arrays, updated state or None)."""
    tabs = [table_bits(t) for t in tables]
    st = None if state is None else state.detach().cpu().numpy().copy()
    oracle.backward(tabs, [DT_NAME[t.dtype] for t in tables], np_index(indices), np_index(offsets),
                    B, grad.detach().cpu().numpy(), optimizer, lr, eps=eps,
                    weights=None if weights is None else np_index(weights), pooling=pooling,
                    state=st)
    return tabs, st


def touched_rows(tables, indices, offsets, B):
    """Per table, a bool mask of the rows at least one valid lookup names."""
    rows = [int(t.shape[0]) for t in tables]
    keys, _ = oracle.make_keys(rows, np_index(indices), np_index(offsets), B)
    rowbase = np.concatenate([[0], np.cumsum(rows)])
    masks = []
    for t in range(len(tables)):
        k = keys[(keys >= rowbase[t]) & (keys < rowbase[t + 1])] - rowbase[t]
        m = np.zeros(rows[t], dtype=bool)
        m[k] = True
        masks.append(m)
    return masks


def assert_tables_match(gpu_tables, ref_bits, before_bits, touched, what=""):
    """Rows without lookups are bit-identical to before; looked-up rows match
    the oracle within the storage dtype's tolerance."""
    for t, (g, r, b, m) in enumerate(zip(gpu_tables, ref_bits, before_bits, touched)):
        name = DT_NAME[g.dtype]
        gb = table_bits(g)
        np.testing.assert_array_equal(gb[~m], b[~m], err_msg=f"{what} table {t}: rows without lookups changed")
        np.testing.assert_array_equal(r[~m], b[~m], err_msg=f"{what} table {t}: oracle changed an untouched row")
        tol = FP32_TOL if name == "f32" else LOWP_TOL
        assert_close(oracle.decode(name, gb[m]), oracle.decode(name, r[m]), what=f"{what} table {t}", **tol)
