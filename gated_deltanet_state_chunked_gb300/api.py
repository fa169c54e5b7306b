"""Python binding of libgdn.so: same names as the C ABI, argument marshalling only.

PyTorch supplies device memory and streams; every step of the computation
runs in the library's CUDA kernels.  There is no CPU fallback: these
functions raise when the library is missing or a tensor is not on a CUDA
device.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

_DTYPE = {torch.float32: _lib.GDN_F32, torch.bfloat16: _lib.GDN_BF16}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _need_cuda(name, t, dtype=None, shape=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def gdn_replay(q, k, v, g, beta, cu_seqlens, S0=None, *, O_out=None, S_out=None, l2norm_qk=True,
               scale=1.0, state_only=False, precise=False, scalar_decay=False, stream=None):
    """Rebuild the recurrent state of each packed replay tail (see gdn.h).

    q, k: [T, h_k, d_k]; v: [T, h_v, d_v] (all bf16 or all fp32); g, beta: fp32
    [T, h_v]; cu_seqlens: int32 [n + 1] on the device; S0: fp32 [n, h_v, d_v, d_k]
    or None.  Returns (O, S): O [T, h_v, d_v] in the input dtype (None when
    ``state_only``) and S fp32 [n, h_v, d_v, d_k]."""
    lib = _lib.load()
    T, h_k, d_k = k.shape
    h_v, d_v = v.shape[1], v.shape[2]
    n = cu_seqlens.shape[0] - 1
    dt = q.dtype
    if dt not in _DTYPE:
        raise ValueError(f"unsupported dtype {dt}")
    _need_cuda("q", q, dt, (T, h_k, d_k))
    _need_cuda("k", k, dt)
    _need_cuda("v", v, dt, (T, h_v, d_v))
    _need_cuda("g", g, torch.float32, (T, h_v))
    _need_cuda("beta", beta, torch.float32, (T, h_v))
    _need_cuda("cu_seqlens", cu_seqlens, torch.int32)
    _need_cuda("S0", S0, torch.float32, (n, h_v, d_v, d_k))
    if S_out is None:
        S_out = torch.empty((n, h_v, d_v, d_k), dtype=torch.float32, device=k.device)
    _need_cuda("S_out", S_out, torch.float32, (n, h_v, d_v, d_k))
    if not state_only:
        if O_out is None:
            O_out = torch.empty((T, h_v, d_v), dtype=dt, device=k.device)
        _need_cuda("O_out", O_out, dt, (T, h_v, d_v))
    else:
        O_out = None
    flags = (_lib.GDN_QK_L2NORM if l2norm_qk else 0) | (_lib.GDN_STATE_ONLY if state_only else 0) \
        | (_lib.GDN_PRECISE if precise else 0) | (_lib.GDN_SCALAR_DECAY if scalar_decay else 0)
    dims = _lib.GdnDims(n, T, h_k, h_v, d_k, d_v, _DTYPE[dt], flags, float(scale))
    rc = lib.gdn_replay(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens),
                        _ptr(S0), _ptr(O_out), _ptr(S_out), _stream_handle(stream, k.device))
    _lib.check(rc, "gdn_replay")
    return O_out, S_out


def gdn_replay_noalloc(q, k, v, g, beta, cu_seqlens, S0, O_out, S_out, *, l2norm_qk=True, scale=1.0,
                       state_only=False, precise=False, scalar_decay=False, stream=None):
    """gdn_replay for callers that cannot allocate device memory at call time.

    Same arguments and results as gdn_replay, except that the outputs O_out
    (None with ``state_only``) and S_out must be passed in: neither this
    wrapper nor the library allocates anything.  The library's scratch is a
    96 MiB static device array shared by all calls, so calls that overlap on
    the GPU race; larger problems raise GdnError(GDN_ERR_NOMEM)."""
    lib = _lib.load()
    T, h_k, d_k = k.shape
    h_v, d_v = v.shape[1], v.shape[2]
    n = cu_seqlens.shape[0] - 1
    dt = q.dtype
    if dt not in _DTYPE:
        raise ValueError(f"unsupported dtype {dt}")
    _need_cuda("q", q, dt, (T, h_k, d_k))
    _need_cuda("k", k, dt)
    _need_cuda("v", v, dt, (T, h_v, d_v))
    _need_cuda("g", g, torch.float32, (T, h_v))
    _need_cuda("beta", beta, torch.float32, (T, h_v))
    _need_cuda("cu_seqlens", cu_seqlens, torch.int32)
    _need_cuda("S0", S0, torch.float32, (n, h_v, d_v, d_k))
    if S_out is None or (O_out is None and not state_only):
        raise ValueError("gdn_replay_noalloc needs caller-provided outputs")
    _need_cuda("S_out", S_out, torch.float32, (n, h_v, d_v, d_k))
    if not state_only:
        _need_cuda("O_out", O_out, dt, (T, h_v, d_v))
    else:
        O_out = None
    flags = (_lib.GDN_QK_L2NORM if l2norm_qk else 0) | (_lib.GDN_STATE_ONLY if state_only else 0) \
        | (_lib.GDN_PRECISE if precise else 0) | (_lib.GDN_SCALAR_DECAY if scalar_decay else 0)
    dims = _lib.GdnDims(n, T, h_k, h_v, d_k, d_v, _DTYPE[dt], flags, float(scale))
    rc = lib.gdn_replay_noalloc(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                _ptr(cu_seqlens), _ptr(S0), _ptr(O_out), _ptr(S_out), _stream_handle(stream, k.device))
    _lib.check(rc, "gdn_replay_noalloc")
    return O_out, S_out


def gdn_chunk_operator(k, g, beta, v, cu_seqlens=None, *, T_out=None, Slocal_out=None, l2norm_qk=True,
                       scalar_decay=False, stream=None):
    """(T_C, S_local) of each chunk (range of cu_seqlens, or all tokens when None).
    ``scalar_decay``: the scalar-transition family (T_C is then a scaled identity).
    Returns T fp32 [n, h_v, d_k, d_k] and S_local fp32 [n, h_v, d_v, d_k]."""
    lib = _lib.load()
    T, h_k, d_k = k.shape
    h_v, d_v = v.shape[1], v.shape[2]
    n = 1 if cu_seqlens is None else cu_seqlens.shape[0] - 1
    dt = k.dtype
    if dt not in _DTYPE:
        raise ValueError(f"unsupported dtype {dt}")
    _need_cuda("k", k, dt)
    _need_cuda("v", v, dt, (T, h_v, d_v))
    _need_cuda("g", g, torch.float32, (T, h_v))
    _need_cuda("beta", beta, torch.float32, (T, h_v))
    _need_cuda("cu_seqlens", cu_seqlens, torch.int32)
    if T_out is None:
        T_out = torch.empty((n, h_v, d_k, d_k), dtype=torch.float32, device=k.device)
    if Slocal_out is None:
        Slocal_out = torch.empty((n, h_v, d_v, d_k), dtype=torch.float32, device=k.device)
    _need_cuda("T_out", T_out, torch.float32, (n, h_v, d_k, d_k))
    _need_cuda("Slocal_out", Slocal_out, torch.float32, (n, h_v, d_v, d_k))
    flags = (_lib.GDN_QK_L2NORM if l2norm_qk else 0) | (_lib.GDN_SCALAR_DECAY if scalar_decay else 0)
    dims = _lib.GdnDims(n, T, h_k, h_v, d_k, d_v, _DTYPE[dt], flags, 1.0)
    rc = lib.gdn_chunk_operator(ctypes.byref(dims), _ptr(k), _ptr(g), _ptr(beta), _ptr(v), _ptr(cu_seqlens),
                                _ptr(T_out), _ptr(Slocal_out), _stream_handle(stream, k.device))
    _lib.check(rc, "gdn_chunk_operator")
    return T_out, Slocal_out


def gdn_compose(T_list, Slocal_list, S_in=None, *, S_out=None, stream=None):
    """S <- S T_j^T + S_local_j for j = 1..K.  T_list[j]: fp32 [h, d_k, d_k];
    Slocal_list[j]: fp32 [h, d_v, d_k]; S_in: [h, d_v, d_k] or None."""
    lib = _lib.load()
    K = len(T_list)
    if len(Slocal_list) != K:
        raise ValueError("T_list and Slocal_list differ in length")
    ref = Slocal_list[0] if K else S_in
    if ref is None:
        raise ValueError("need at least one chunk or an entering state")
    h, d_v, d_k = ref.shape
    for j in range(K):
        _need_cuda(f"T[{j}]", T_list[j], torch.float32, (h, d_k, d_k))
        _need_cuda(f"Slocal[{j}]", Slocal_list[j], torch.float32, (h, d_v, d_k))
    _need_cuda("S_in", S_in, torch.float32, (h, d_v, d_k))
    if S_out is None:
        S_out = torch.empty((h, d_v, d_k), dtype=torch.float32, device=ref.device)
    _need_cuda("S_out", S_out, torch.float32, (h, d_v, d_k))
    Tp = (ctypes.c_void_p * max(K, 1))(*[t.data_ptr() for t in T_list])
    Sp = (ctypes.c_void_p * max(K, 1))(*[s.data_ptr() for s in Slocal_list])
    dims = _lib.GdnDims(1, 0, h, h, d_k, d_v, _lib.GDN_F32, 0, 1.0)
    rc = lib.gdn_compose(ctypes.byref(dims), K, ctypes.cast(Tp, ctypes.c_void_p), ctypes.cast(Sp, ctypes.c_void_p),
                         _ptr(S_in), _ptr(S_out), _stream_handle(stream, ref.device))
    _lib.check(rc, "gdn_compose")
    return S_out


def gdn_get_status(stream=None, device=None):
    """Synchronise the stream; raise GdnError if the device recorded an error."""
    lib = _lib.load()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    rc = lib.gdn_get_status(_stream_handle(stream, dev))
    _lib.check(rc, "gdn_get_status")


def gdn_workspace_bytes(n_seqs, total_tokens, h_k, h_v, d_k, d_v, dtype=torch.bfloat16, flags=0) -> int:
    lib = _lib.load()
    dims = _lib.GdnDims(n_seqs, total_tokens, h_k, h_v, d_k, d_v, _DTYPE[dtype], flags, 1.0)
    return int(lib.gdn_workspace_bytes(ctypes.byref(dims)))


def gdn_set_stage_event(event) -> None:
    """Have this thread's next tensor-core gdn_replay record ``event`` (a
    torch.cuda.Event) between its prep and scan kernels (measurement hook)."""
    lib = _lib.load()
    if event is not None and event.cuda_event == 0:
        raise ValueError("record-able torch.cuda.Event expected")
    lib.gdn_set_stage_event(ctypes.c_void_p(event.cuda_event if event is not None else 0))


def gdn_set_wait_limit_ns(ns: int) -> None:
    """Bound of the device-side waits of this thread's next gdn_compose call (test hook of the
    timeout path; 0 makes a wait give up unless its event has already happened)."""
    _lib.load().gdn_set_wait_limit_ns(int(ns))
