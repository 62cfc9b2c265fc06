"""Table-batched embedding (TBE) on GB300: Python binding of ``libtbe_gb300.so``.

The functions here carry the names of the C ABI in ``include/tbe.h`` and only
marshal arguments: torch tensors become device pointers, the current torch
stream becomes the ``stream`` argument, and a nonzero status raises
:class:`TBEError`.  Every step of the operator runs in the library's CUDA
kernels.  If the library has not been built, importing works but the first
call raises; there is no other implementation to fall back on.
"""

from __future__ import annotations

import ctypes
import os
import re
from typing import List, Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtbe_gb300.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "tbe.h")

TBE_OK = 0
TBE_ERR_INVALID_ARG = -1
TBE_ERR_UNSUPPORTED = -2
TBE_ERR_WORKSPACE_TOO_SMALL = -3
TBE_ERR_CUDA = -4
TBE_ERR_INDEX_OOB = -5
TBE_ERR_BAD_OFFSETS = -6
TBE_ERR_TIMEOUT = -7
TBE_ERR_NO_MEMORY = -8

TBE_F32, TBE_F16, TBE_BF16 = 0, 1, 2
TBE_I32, TBE_I64 = 0, 1
TBE_POOL_SUM, TBE_POOL_MEAN = 0, 1
TBE_OPT_SGD, TBE_OPT_ROWWISE_ADAGRAD = 1, 2
TBE_FLAG_NO_HISTOGRAM = 0x1
TBE_FLAG_FORCE_HISTOGRAM = 0x2
TBE_FLAG_SORTED_BACKWARD = 0x4
TBE_FLAG_LENGTH_ORDER = 0x8

PATH_NAMES = {0: "gather", 1: "gather_elementwise", 2: "histogram"}

_DTYPES = {torch.float32: TBE_F32, torch.float16: TBE_F16, torch.bfloat16: TBE_BF16}
_POOL = {"sum": TBE_POOL_SUM, "mean": TBE_POOL_MEAN}


class TBEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {tbe_strerror(code)} ({code})")


class _Table(ctypes.Structure):
    _fields_ = [("rows", ctypes.c_int64), ("dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("data", ctypes.c_void_p)]


class _Optimizer(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("lr", ctypes.c_float), ("eps", ctypes.c_float),
                ("state", ctypes.c_void_p)]


class WorkspaceLayout(ctypes.Structure):
    _fields_ = [("sorted_keys", ctypes.c_uint64), ("sorted_vals", ctypes.c_uint64),
                ("uniq", ctypes.c_uint64), ("runstart", ctypes.c_uint64),
                ("num_unique", ctypes.c_uint64), ("total_bytes", ctypes.c_uint64)]


_lib = None


def library_path() -> str:
    return LIB_PATH


def load_library():
    """Load ``libtbe_gb300.so``; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, u32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_float
    sig = {
        "tbe_create": ([ctypes.POINTER(_Table), i32, i32, u32, ctypes.POINTER(P)], ctypes.c_int),
        "tbe_destroy": ([P], None),
        "tbe_forward": ([P, P, P, i32, i64, i32, P, P, P], ctypes.c_int),
        "tbe_backward_workspace_bytes": ([P, i64, i32], ctypes.c_size_t),
        "tbe_backward_workspace_layout": ([P, i64, i32, ctypes.POINTER(WorkspaceLayout)], ctypes.c_int),
        "tbe_backward_prepare": ([P, P, P, i32, i64, i32, P, P, ctypes.c_size_t, P], ctypes.c_int),
        "tbe_forward_prepare": ([P, P, P, i32, i64, i32, P, P, P, ctypes.c_size_t, P], ctypes.c_int),
        "tbe_backward_apply": ([P, i64, i32, P, ctypes.POINTER(_Optimizer), P, ctypes.c_size_t, P],
                               ctypes.c_int),
        "tbe_backward_sgd": ([P, P, P, i32, i64, i32, P, P, f32, P, ctypes.c_size_t, P], ctypes.c_int),
        "tbe_backward_rowwise_adagrad": ([P, P, P, i32, i64, i32, P, P, P, f32, f32, P,
                                          ctypes.c_size_t, P], ctypes.c_int),
        "tbe_backward_sgd_noalloc": ([P, P, P, i32, i64, i32, P, P, f32, P], ctypes.c_int),
        "tbe_per_sample_weight_grad": ([P, P, P, i32, i64, i32, P, P, P], ctypes.c_int),
        "tbe_get_error": ([P, P], ctypes.c_int),
        "tbe_strerror": ([ctypes.c_int], ctypes.c_char_p),
        "tbe_last_cuda_error": ([], ctypes.c_int),
        "tbe_table_paths": ([P, ctypes.POINTER(i32)], ctypes.c_int),
        "tbe_table_backward_paths": ([P, ctypes.POINTER(i32)], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def declared_functions() -> List[str]:
    """Names of the functions include/tbe.h declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tbe_[a-z0-9_]+)\s*\(", text)))


def _check(rc: int, where: str):
    if rc != TBE_OK:
        if rc == TBE_ERR_CUDA:
            where = f"{where} (cudaError_t {load_library().tbe_last_cuda_error()})"
        raise TBEError(rc, where)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _index_dtype(indices: torch.Tensor, offsets: torch.Tensor) -> int:
    if indices.dtype != offsets.dtype or indices.dtype not in (torch.int32, torch.int64):
        raise ValueError("indices and offsets must share dtype int32 or int64")
    return TBE_I64 if indices.dtype == torch.int64 else TBE_I32


def tbe_strerror(code: int) -> str:
    try:
        return load_library().tbe_strerror(code).decode()
    except RuntimeError:
        return f"status {code}"


class Handle:
    """A created TBE handle.  Keeps the tables alive; ``close()`` (or garbage
    collection) calls tbe_destroy."""

    def __init__(self, ptr: ctypes.c_void_p, tables: Sequence[torch.Tensor], pooling: str):
        self._ptr = ptr
        self.tables = list(tables)
        self.pooling = pooling
        self.dims = [int(t.shape[1]) for t in tables]
        self.rows = [int(t.shape[0]) for t in tables]
        self.total_dim = sum(self.dims)
        self.total_rows = sum(self.rows)

    @property
    def ptr(self):
        if self._ptr is None:
            raise RuntimeError("handle already destroyed")
        return self._ptr

    def close(self):
        if self._ptr is not None and _lib is not None:
            _lib.tbe_destroy(self._ptr)
        self._ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def tbe_create(tables: Sequence[torch.Tensor], pooling: str = "sum", flags: int = 0) -> Handle:
    """Tables: CUDA tensors [rows, dim] (fp32/fp16/bf16), updated in place by backward."""
    lib = load_library()
    arr = (_Table * len(tables))()
    for i, t in enumerate(tables):
        if t.dim() != 2 or t.dtype not in _DTYPES:
            raise ValueError("tables must be 2-D fp32/fp16/bf16 CUDA tensors")
        if not t.is_contiguous():
            raise ValueError("tables must be contiguous (row-major, rows packed)")
        arr[i] = _Table(t.shape[0], t.shape[1], _DTYPES[t.dtype], _ptr(t))
    out = ctypes.c_void_p()
    _check(lib.tbe_create(arr, len(tables), _POOL[pooling], flags, ctypes.byref(out)), "tbe_create")
    return Handle(out, tables, pooling)


def tbe_destroy(h: Handle):
    h.close()


def tbe_table_paths(h: Handle) -> List[str]:
    buf = (ctypes.c_int32 * len(h.tables))()
    _check(load_library().tbe_table_paths(h.ptr, buf), "tbe_table_paths")
    return [PATH_NAMES[int(x)] for x in buf]


def tbe_backward_paths(h: Handle) -> List[str]:
    """Per table, "dense" (tensor-core H^T . G) or "sorted"."""
    buf = (ctypes.c_int32 * len(h.tables))()
    _check(load_library().tbe_table_backward_paths(h.ptr, buf), "tbe_table_backward_paths")
    return ["dense" if int(x) else "sorted" for x in buf]


def tbe_forward(h: Handle, indices: torch.Tensor, offsets: torch.Tensor, batch_size: int,
                per_sample_weights: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
    lib = load_library()
    if out is None:
        out = torch.empty((batch_size, h.total_dim), dtype=torch.float32, device=offsets.device)
    rc = lib.tbe_forward(h.ptr, _ptr(indices), _ptr(offsets), _index_dtype(indices, offsets),
                         indices.numel(), batch_size, _ptr(per_sample_weights), _ptr(out),
                         _stream(stream))
    _check(rc, "tbe_forward")
    return out


def tbe_per_sample_weight_grad(h: Handle, indices: torch.Tensor, offsets: torch.Tensor, batch_size: int,
                               grad_out: torch.Tensor, grad_weights: Optional[torch.Tensor] = None,
                               stream=None) -> torch.Tensor:
    """dL/dw_i for every lookup; call before the backward pass updates the rows."""
    lib = load_library()
    if grad_weights is None:
        grad_weights = torch.empty(indices.numel(), dtype=torch.float32, device=offsets.device)
    rc = lib.tbe_per_sample_weight_grad(h.ptr, _ptr(indices), _ptr(offsets), _index_dtype(indices, offsets),
                                        indices.numel(), batch_size, _ptr(grad_out), _ptr(grad_weights),
                                        _stream(stream))
    _check(rc, "tbe_per_sample_weight_grad")
    return grad_weights


def tbe_backward_workspace_bytes(h: Handle, num_indices: int, batch_size: int) -> int:
    return int(load_library().tbe_backward_workspace_bytes(h.ptr, num_indices, batch_size))


def tbe_backward_workspace_layout(h: Handle, num_indices: int, batch_size: int) -> WorkspaceLayout:
    out = WorkspaceLayout()
    _check(load_library().tbe_backward_workspace_layout(h.ptr, num_indices, batch_size,
                                                        ctypes.byref(out)),
           "tbe_backward_workspace_layout")
    return out


def make_workspace(h: Handle, num_indices: int, batch_size: int, device=None) -> torch.Tensor:
    n = tbe_backward_workspace_bytes(h, num_indices, batch_size)
    return torch.empty(n, dtype=torch.uint8, device=device or h.tables[0].device)


def tbe_backward_prepare(h: Handle, indices, offsets, batch_size: int, workspace: torch.Tensor,
                         per_sample_weights=None, stream=None):
    rc = load_library().tbe_backward_prepare(
        h.ptr, _ptr(indices), _ptr(offsets), _index_dtype(indices, offsets), indices.numel(),
        batch_size, _ptr(per_sample_weights), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "tbe_backward_prepare")


def tbe_forward_prepare(h: Handle, indices, offsets, batch_size: int, workspace: torch.Tensor,
                        per_sample_weights=None, out: Optional[torch.Tensor] = None, stream=None):
    """Forward pass and backward preparation of one batch, run side by side."""
    if out is None:
        out = torch.empty((batch_size, h.total_dim), dtype=torch.float32, device=offsets.device)
    rc = load_library().tbe_forward_prepare(
        h.ptr, _ptr(indices), _ptr(offsets), _index_dtype(indices, offsets), indices.numel(),
        batch_size, _ptr(per_sample_weights), _ptr(out), _ptr(workspace), workspace.numel(),
        _stream(stream))
    _check(rc, "tbe_forward_prepare")
    return out


def tbe_backward_apply(h: Handle, num_indices: int, batch_size: int, grad_out: torch.Tensor,
                       workspace: torch.Tensor, optimizer: str = "sgd", lr: float = 0.01,
                       eps: float = 0.0, state: Optional[torch.Tensor] = None, stream=None):
    kind = TBE_OPT_SGD if optimizer == "sgd" else TBE_OPT_ROWWISE_ADAGRAD
    opt = _Optimizer(kind, lr, eps, _ptr(state))
    rc = load_library().tbe_backward_apply(h.ptr, num_indices, batch_size, _ptr(grad_out),
                                           ctypes.byref(opt), _ptr(workspace), workspace.numel(),
                                           _stream(stream))
    _check(rc, "tbe_backward_apply")


def tbe_backward_sgd(h: Handle, indices, offsets, batch_size: int, grad_out, lr: float,
                     workspace: torch.Tensor, per_sample_weights=None, stream=None):
    rc = load_library().tbe_backward_sgd(
        h.ptr, _ptr(indices), _ptr(offsets), _index_dtype(indices, offsets), indices.numel(),
        batch_size, _ptr(per_sample_weights), _ptr(grad_out), lr, _ptr(workspace),
        workspace.numel(), _stream(stream))
    _check(rc, "tbe_backward_sgd")


def tbe_backward_rowwise_adagrad(h: Handle, indices, offsets, batch_size: int, grad_out,
                                 state: torch.Tensor, lr: float, eps: float,
                                 workspace: torch.Tensor, per_sample_weights=None, stream=None):
    rc = load_library().tbe_backward_rowwise_adagrad(
        h.ptr, _ptr(indices), _ptr(offsets), _index_dtype(indices, offsets), indices.numel(),
        batch_size, _ptr(per_sample_weights), _ptr(grad_out), _ptr(state), lr, eps,
        _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "tbe_backward_rowwise_adagrad")


def tbe_backward_sgd_noalloc(h: Handle, indices, offsets, batch_size: int, grad_out, lr: float,
                             per_sample_weights=None, stream=None):
    """tbe_backward_sgd with the library's static 32 MiB workspace: for callers
    that cannot allocate device memory for a workspace (see include/tbe.h)."""
    rc = load_library().tbe_backward_sgd_noalloc(
        h.ptr, _ptr(indices), _ptr(offsets), _index_dtype(indices, offsets), indices.numel(),
        batch_size, _ptr(per_sample_weights), _ptr(grad_out), lr, _stream(stream))
    _check(rc, "tbe_backward_sgd_noalloc")


def tbe_get_error(h: Handle, stream=None) -> int:
    return int(load_library().tbe_get_error(h.ptr, _stream(stream)))


__all__ = [n for n in dir() if n.startswith("tbe_") or n.startswith("TBE_")] + [
    "Handle", "TBEError", "WorkspaceLayout", "load_library", "declared_functions",
    "make_workspace", "library_path"]
