"""The C-ABI library loads, exports what include/gdn.h declares, and rejects
bad arguments on the host before touching a GPU (no compute call is made)."""
import ctypes

import pytest

from gated_deltanet_state_chunked_gb300 import _lib


@pytest.fixture(scope="module")
def lib():
    return _lib.load(build=True)


def test_exports_every_declared_symbol(lib):
    names = _lib.header_functions()
    assert set(names) >= {"gdn_replay", "gdn_chunk_operator", "gdn_compose", "gdn_get_status",
                          "gdn_last_error", "gdn_workspace_bytes", "gdn_abi_version"}
    for n in names:
        assert hasattr(lib, n), n
    assert set(_lib.SIGNATURES) >= set(names)


def test_abi_version(lib):
    assert lib.gdn_abi_version() == 1


def _dims(**kw):
    d = dict(n_seqs=1, total_tokens=64, h_k=2, h_v=4, d_k=64, d_v=64, dtype=_lib.GDN_BF16,
             flags=_lib.GDN_QK_L2NORM, scale=1.0)
    d.update(kw)
    return _lib.GdnDims(**d)


A16 = ctypes.c_void_p(1 << 20)        # 16-byte aligned fake addresses (never dereferenced:
A16b = ctypes.c_void_p((1 << 20) + 256)  # every call below fails its host checks first)
MIS = ctypes.c_void_p((1 << 20) + 8)


def _replay(lib, dims, q=A16, O=A16b, S0=None, cu=A16):
    return lib.gdn_replay(ctypes.byref(dims) if dims is not None else None, q, A16, A16, A16, A16, cu, S0, O, A16b, None)


def test_null_dims_is_arg_error(lib):
    assert _replay(lib, None) == _lib.GDN_ERR_ARG
    assert b"dims" in lib.gdn_last_error()


@pytest.mark.parametrize("kw,code", [
    (dict(h_v=3), _lib.GDN_ERR_SHAPE),
    (dict(h_k=0), _lib.GDN_ERR_ARG),
    (dict(d_k=12), _lib.GDN_ERR_UNSUPPORTED),
    (dict(d_v=256), _lib.GDN_ERR_UNSUPPORTED),
    (dict(dtype=7), _lib.GDN_ERR_UNSUPPORTED),
    (dict(flags=64), _lib.GDN_ERR_ARG),
    (dict(n_seqs=-1), _lib.GDN_ERR_ARG),
])
def test_bad_dims_rejected(lib, kw, code):
    assert _replay(lib, _dims(**kw)) == code
    assert lib.gdn_last_error() != b""


def test_missing_output_rejected(lib):
    assert _replay(lib, _dims(), O=None) == _lib.GDN_ERR_ARG
    assert _replay(lib, _dims(), cu=None) == _lib.GDN_ERR_ARG


def test_misaligned_pointer_rejected(lib):
    assert _replay(lib, _dims(), q=MIS) == _lib.GDN_ERR_ALIGN
    assert _replay(lib, _dims(), S0=MIS) == _lib.GDN_ERR_ALIGN


def test_empty_batch_is_a_no_op(lib):
    assert _replay(lib, _dims(n_seqs=0)) == _lib.GDN_OK


def test_chunk_operator_and_compose_checks(lib):
    d = _dims()
    assert lib.gdn_chunk_operator(ctypes.byref(_dims(n_seqs=2)), A16, A16, A16, A16, None, A16, A16b, None) \
        == _lib.GDN_ERR_ARG
    assert lib.gdn_chunk_operator(ctypes.byref(d), A16, A16, A16, A16, None, None, A16b, None) == _lib.GDN_ERR_ARG
    arr = (ctypes.c_void_p * 1)(A16.value)
    assert lib.gdn_compose(ctypes.byref(d), 1, arr, arr, None, A16, None) == _lib.GDN_ERR_ARG  # aliasing
    assert lib.gdn_compose(ctypes.byref(d), -1, arr, arr, None, A16b, None) == _lib.GDN_ERR_ARG
    assert lib.gdn_compose(ctypes.byref(d), 1000, arr, arr, None, A16b, None) == _lib.GDN_ERR_ARG
    mis = (ctypes.c_void_p * 1)(MIS.value)
    assert lib.gdn_compose(ctypes.byref(d), 1, mis, arr, None, A16b, None) == _lib.GDN_ERR_ALIGN


def test_workspace_query_needs_no_gpu(lib):
    assert lib.gdn_workspace_bytes(ctypes.byref(_dims())) >= 0
