"""CPU oracle for table-batched embedding (TBE): TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct statement of what the operator computes,
written in C (``tbe_oracle.c``) in double precision, with this ctypes
wrapper.  Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it.  It shares no code with the CUDA library
under ``recommender_sparse_embeddings_gb300/`` and the library never calls it.

Parity pins (tests/test_oracle_pins.py) tie each function here to something
other than itself: the worked call on the FBTriton integration page, torch's
CPU ``embedding_bag`` and autograd in fp64, a dense matrix formulation,
numpy's stable argsort and unique, numpy/torch float conversions, and
torch.optim.SGD / torch.optim.Adagrad on the cases where row-wise Adagrad
reduces to the element-wise one.  Row-wise Adagrad itself and the
out-of-range-index rule are readings (the pages do not define them); they are
pinned only through those special cases.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tbe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libtbe_oracle.so")
# The timing build: the same source at -O3 with OpenMP, whose parallel loops
# (bags of the forward pass, runs of the backward pass) run on the host's
# cores.  Each bag's and each run's sums are the same sequence of additions
# as in the plain build; only the CPU baseline of bench.py loads it.
_OMP_LIB_PATH = os.path.join(_HERE, "libtbe_oracle_omp.so")

DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2}
OPT_CODES = {"none": 0, "sgd": 1, "adagrad": 2, "rowwise_adagrad": 2}

_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/libtbe_oracle.so`` (gcc, -O2).

    ``-ffp-contract=off`` keeps every multiply and add separately rounded so
    the double-precision results are the same on x86 and Arm hosts."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-ffp-contract=off", "-Wall", "-Wextra", "-Wno-unknown-pragmas", "-o", tmp,
                               _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def build_timing(force: bool = False) -> str:
    """Compile the timing build ``oracle/libtbe_oracle_omp.so`` (gcc -O3
    -fopenmp, contraction still off)."""
    if force or not os.path.exists(_OMP_LIB_PATH) or (
            os.path.getmtime(_OMP_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _OMP_LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O3", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _OMP_LIB_PATH)
    return _OMP_LIB_PATH


_timing = False


def use_timing_build(threads: int) -> int:
    """Route the calls below to the timing build with `threads` threads;
    returns the thread count in effect.  (For bench.py's CPU baseline.)"""
    global _timing, _lib
    if not _timing:
        build_timing()
        _timing, _lib = True, None
    return int(_load().oracle_set_threads(int(threads)))


def use_plain_build() -> None:
    """Route the calls back to the plain (pinned, one-thread) build."""
    global _timing, _lib
    if _timing:
        _timing, _lib = False, None


def _load():
    global _lib
    if _lib is None:
        if _timing:
            lib = ctypes.CDLL(_OMP_LIB_PATH)
        else:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
        lib.oracle_set_threads.argtypes = [ctypes.c_int32]
        lib.oracle_set_threads.restype = ctypes.c_int
        P = ctypes.c_void_p
        i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        lib.oracle_forward.argtypes = [i32, P, P, P, P, i32, i32, P, P, i64, P, i32, P, P]
        lib.oracle_forward.restype = ctypes.c_int
        lib.oracle_make_keys.argtypes = [i32, P, i32, i32, P, P, i64, P, P]
        lib.oracle_make_keys.restype = ctypes.c_int
        lib.oracle_sort_rle.argtypes = [P, i64, P, P, P, P, P]
        lib.oracle_sort_rle.restype = ctypes.c_int64
        lib.oracle_backward.argtypes = [i32, P, P, P, P, i32, i32, P, P, i64, P, i32, P, i32,
                                        f32, f32, P, P, P, P]
        lib.oracle_backward.restype = ctypes.c_int
        lib.oracle_weight_grad.argtypes = [i32, P, P, P, P, i32, i32, P, P, i64, i32, P, P]
        lib.oracle_weight_grad.restype = ctypes.c_int
        lib.oracle_round.argtypes = [i32, P, i64, P]
        lib.oracle_round.restype = None
        lib.oracle_decode.argtypes = [i32, P, i64, P]
        lib.oracle_decode.restype = None
        _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _table_bits(w: np.ndarray, dtype: str) -> np.ndarray:
    """Tables are float32 arrays (f32) or uint16/float16 arrays of raw bits."""
    if dtype == "f32":
        if w.dtype != np.float32:
            raise TypeError("f32 table must be a float32 array")
        return np.ascontiguousarray(w)
    if w.dtype == np.float16:
        w = w.view(np.uint16)
    if w.dtype != np.uint16:
        raise TypeError(f"{dtype} table must hold raw 16-bit patterns (uint16)")
    return np.ascontiguousarray(w)


def _index_arrays(indices, offsets):
    indices = np.ascontiguousarray(indices)
    offsets = np.ascontiguousarray(offsets)
    if indices.dtype != offsets.dtype or indices.dtype not in (np.int32, np.int64):
        raise TypeError("indices and offsets must share dtype int32 or int64")
    return indices, offsets, int(indices.dtype == np.int64)


def _table_meta(tables, dtypes):
    rows = np.array([w.shape[0] for w in tables], dtype=np.int64)
    dims = np.array([w.shape[1] for w in tables], dtype=np.int32)
    codes = np.array([DTYPE_CODES[d] for d in dtypes], dtype=np.int32)
    return rows, dims, codes


def forward(tables: Sequence[np.ndarray], dtypes: Sequence[str], indices, offsets, B: int,
            weights=None, pooling: str = "sum"):
    """Pooled lookup of every bag of every table.

    Returns (out [B, sum D] float32, number of skipped out-of-range lookups)."""
    lib = _load()
    tabs = [_table_bits(w, d) for w, d in zip(tables, dtypes)]
    rows, dims, codes = _table_meta(tabs, dtypes)
    indices, offsets, is64 = _index_arrays(indices, offsets)
    T = len(tabs)
    if offsets.shape[0] != T * B + 1:
        raise ValueError("offsets must have T*B+1 entries")
    ptrs = (ctypes.c_void_p * T)(*[w.ctypes.data for w in tabs])
    w = None if weights is None else np.ascontiguousarray(weights, dtype=np.float32)
    out = np.zeros((B, int(dims.sum())), dtype=np.float32)
    skipped = ctypes.c_int64(0)
    rc = lib.oracle_forward(T, _ptr(rows), _ptr(dims), _ptr(codes), ptrs, B, is64,
                            _ptr(indices), _ptr(offsets), indices.shape[0], _ptr(w),
                            int(pooling == "mean"), _ptr(out), ctypes.byref(skipped))
    if rc:
        raise OracleError(f"oracle_forward failed: {rc}")
    return out, int(skipped.value)


def weight_grad(tables: Sequence[np.ndarray], dtypes: Sequence[str], indices, offsets, B: int, grad_out,
                pooling: str = "sum"):
    """dL/dw_i for every lookup (0 for skipped ones), given G = dL/dout."""
    lib = _load()
    tabs = [_table_bits(w, d) for w, d in zip(tables, dtypes)]
    rows, dims, codes = _table_meta(tabs, dtypes)
    indices, offsets, is64 = _index_arrays(indices, offsets)
    T = len(tabs)
    if offsets.shape[0] != T * B + 1:
        raise ValueError("offsets must have T*B+1 entries")
    g = np.ascontiguousarray(grad_out, dtype=np.float32)
    if g.shape != (B, int(dims.sum())):
        raise ValueError("grad_out must be [B, sum of dims]")
    ptrs = (ctypes.c_void_p * T)(*[w.ctypes.data for w in tabs])
    out = np.zeros(indices.shape[0], dtype=np.float32)
    rc = lib.oracle_weight_grad(T, _ptr(rows), _ptr(dims), _ptr(codes), ptrs, B, is64, _ptr(indices),
                                _ptr(offsets), indices.shape[0], int(pooling == "mean"), _ptr(g), _ptr(out))
    if rc:
        raise OracleError(f"oracle_weight_grad failed: {rc}")
    return out


def make_keys(rows: Sequence[int], indices, offsets, B: int):
    """Transpose step: (key per lookup, flat bag id per lookup), both int64."""
    lib = _load()
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    indices, offsets, is64 = _index_arrays(indices, offsets)
    N = indices.shape[0]
    keys = np.empty(N, dtype=np.int64)
    bag = np.empty(N, dtype=np.int64)
    rc = lib.oracle_make_keys(len(rows), _ptr(rows), B, is64, _ptr(indices), _ptr(offsets), N,
                              _ptr(keys), _ptr(bag))
    if rc:
        raise OracleError(f"oracle_make_keys failed: {rc}")
    return keys, bag


def sort_rle(keys):
    """Stable sort of keys (values = positions) and run-length encoding."""
    lib = _load()
    keys = np.ascontiguousarray(keys, dtype=np.int64)
    N = keys.shape[0]
    sk = np.empty(N, dtype=np.int64)
    sp = np.empty(N, dtype=np.int64)
    uq = np.empty(N, dtype=np.int64)
    rs = np.empty(N, dtype=np.int64)
    rl = np.empty(N, dtype=np.int64)
    U = lib.oracle_sort_rle(_ptr(keys), N, _ptr(sk), _ptr(sp), _ptr(uq), _ptr(rs), _ptr(rl))
    if U < 0:
        raise OracleError(f"oracle_sort_rle failed: {U}")
    return dict(sorted_keys=sk, sorted_pos=sp, uniq=uq[:U].copy(), runstart=rs[:U].copy(),
                runlen=rl[:U].copy())


def backward(tables: Sequence[np.ndarray], dtypes: Sequence[str], indices, offsets, B: int,
             grad_out, optimizer: str, lr: float, eps: float = 0.0, weights=None,
             pooling: str = "sum", state=None, want_row_grads: bool = False):
    """Backward + one optimizer step per touched row, in place on ``tables``
    (and ``state`` for row-wise Adagrad).  Tables must be writable contiguous
    arrays (float32, or uint16 bit patterns for f16/bf16).

    Returns (row_keys, row_grads) when want_row_grads, else None."""
    lib = _load()
    for w, d in zip(tables, dtypes):
        if not w.flags.c_contiguous or not w.flags.writeable:
            raise ValueError("tables must be writable and contiguous (updated in place)")
        _table_bits(w, d)
    tabs = [w.view(np.uint16) if w.dtype == np.float16 else w for w in tables]
    rows, dims, codes = _table_meta(tabs, dtypes)
    indices, offsets, is64 = _index_arrays(indices, offsets)
    T = len(tabs)
    ptrs = (ctypes.c_void_p * T)(*[w.ctypes.data for w in tabs])
    g = np.ascontiguousarray(grad_out, dtype=np.float32)
    if g.shape != (B, int(dims.sum())):
        raise ValueError("grad_out must be [B, sum of dims]")
    w = None if weights is None else np.ascontiguousarray(weights, dtype=np.float32)
    opt = OPT_CODES[optimizer]
    if opt == 2:
        if state is None or state.dtype != np.float32 or state.shape != (int(rows.sum()),):
            raise ValueError("row-wise Adagrad needs a float32 state of sum(rows) entries")
    N = indices.shape[0]
    maxd = int(dims.max())
    rg = np.zeros((N, maxd), dtype=np.float64) if want_row_grads else None
    rk = np.zeros(N, dtype=np.int64) if want_row_grads else None
    nr = ctypes.c_int64(0)
    rc = lib.oracle_backward(T, _ptr(rows), _ptr(dims), _ptr(codes), ptrs, B, is64,
                             _ptr(indices), _ptr(offsets), N, _ptr(w), int(pooling == "mean"),
                             _ptr(g), opt, ctypes.c_float(lr), ctypes.c_float(eps),
                             _ptr(state), _ptr(rg), _ptr(rk), ctypes.byref(nr))
    if rc:
        raise OracleError(f"oracle_backward failed: {rc}")
    if want_row_grads:
        n = int(nr.value)
        return rk[:n].copy(), rg[:n].copy()
    return None


def round_to(dtype: str, x) -> np.ndarray:
    """Round float64 values once, to nearest even, to f32/f16/bf16 storage
    (float32 array for f32, raw uint16 bit patterns otherwise)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float32 if dtype == "f32" else np.uint16)
    lib.oracle_round(DTYPE_CODES[dtype], _ptr(x), x.size, _ptr(out))
    return out


def decode(dtype: str, bits) -> np.ndarray:
    """Exact float64 value of stored f32/f16/bf16 elements."""
    lib = _load()
    bits = np.ascontiguousarray(bits)
    if dtype == "f16" and bits.dtype == np.float16:
        bits = bits.view(np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    lib.oracle_decode(DTYPE_CODES[dtype], _ptr(bits), bits.size, _ptr(out))
    return out
