"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/tbe.h declares, and rejects bad arguments before any
CUDA call."""

import ctypes
import os

import pytest

import recommender_sparse_embeddings_gb300 as tbe

pytestmark = pytest.mark.skipif(not os.path.exists(tbe.library_path()),
                                reason="library not built (run __graft_entry__.build())")


def test_header_declares_the_four_named_calls():
    names = tbe.declared_functions()
    for n in ("tbe_create", "tbe_forward", "tbe_backward_sgd", "tbe_backward_rowwise_adagrad"):
        assert n in names


def test_library_exports_every_declared_function():
    lib = tbe.load_library()
    missing = [n for n in tbe.declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_strerror_covers_every_code():
    codes = [tbe.TBE_OK, tbe.TBE_ERR_INVALID_ARG, tbe.TBE_ERR_UNSUPPORTED,
             tbe.TBE_ERR_WORKSPACE_TOO_SMALL, tbe.TBE_ERR_CUDA, tbe.TBE_ERR_INDEX_OOB,
             tbe.TBE_ERR_BAD_OFFSETS, tbe.TBE_ERR_TIMEOUT, tbe.TBE_ERR_NO_MEMORY]
    texts = [tbe.tbe_strerror(c) for c in codes]
    assert len(set(texts)) == len(texts)
    assert tbe.tbe_strerror(-99) == "unknown error"


def _create(tables, T, pooling=0, flags=0):
    lib = tbe.load_library()
    out = ctypes.c_void_p(123)
    rc = lib.tbe_create(tables, T, pooling, flags, ctypes.byref(out))
    return rc, out


def test_create_rejects_bad_arguments_without_cuda():
    Table = tbe._Table
    good = (Table * 1)(Table(10, 4, tbe.TBE_F32, ctypes.c_void_p(0x1000)))
    assert _create(None, 1)[0] == tbe.TBE_ERR_INVALID_ARG
    assert _create(good, 0)[0] == tbe.TBE_ERR_INVALID_ARG
    rc, out = _create(good, 1, pooling=7)
    assert rc == tbe.TBE_ERR_INVALID_ARG and out.value is None
    assert _create(good, 1, flags=0x80)[0] == tbe.TBE_ERR_INVALID_ARG
    for bad in (Table(0, 4, 0, ctypes.c_void_p(0x1000)), Table(10, 0, 0, ctypes.c_void_p(0x1000)),
                Table(10, 4, 9, ctypes.c_void_p(0x1000)), Table(10, 4, 0, None)):
        assert _create((Table * 1)(bad), 1)[0] == tbe.TBE_ERR_INVALID_ARG
    assert _create((Table * 1)(Table(1 << 31, 4, 0, ctypes.c_void_p(0x1000))), 1)[0] == \
        tbe.TBE_ERR_UNSUPPORTED
    assert _create((Table * 1)(Table(10, 5000, 0, ctypes.c_void_p(0x1000))), 1)[0] == \
        tbe.TBE_ERR_UNSUPPORTED
    big = (Table * 3)(*[Table((1 << 31) - 1, 4, 0, ctypes.c_void_p(0x1000)) for _ in range(3)])
    assert _create(big, 3)[0] == tbe.TBE_ERR_UNSUPPORTED


def test_calls_reject_null_handle():
    lib = tbe.load_library()
    assert lib.tbe_forward(None, None, None, 1, 0, 1, None, None, None) == tbe.TBE_ERR_INVALID_ARG
    assert lib.tbe_backward_workspace_bytes(None, 10, 1) == 0
    assert lib.tbe_get_error(None, None) == tbe.TBE_ERR_INVALID_ARG
    assert lib.tbe_backward_apply(None, 0, 0, None, None, None, 0, None) == tbe.TBE_ERR_INVALID_ARG
    lib.tbe_destroy(None)  # no-op


def test_binding_rejects_tables_that_are_not_packed_rows():
    """A table view whose rows are not packed (an expanded row, a column
    slice) has no row-major layout for the library to index."""
    import torch

    with pytest.raises(ValueError, match="contiguous"):
        tbe.tbe_create([torch.zeros(1, 16).expand(100, 16)])
    with pytest.raises(ValueError, match="contiguous"):
        tbe.tbe_create([torch.zeros(100, 32)[:, :16]])
