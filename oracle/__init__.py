"""fp64 CPU oracle for the Gated DeltaNet tail-replay state rebuild.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline leg
of the benchmark may import this package; the product path never does.  The
arithmetic lives in ``gdn_oracle.c`` (plain C, fp64); this module compiles it
with gcc on first use and marshals numpy arrays.  It shares no code with the
CUDA library.

Functions and the passages they follow:

* :func:`replay` -- "Tail-Replay: Escaping the Curse of Linear Attention in
  Prefix Caching for Hybrid LLMs", section 2 Eq. (1) and section 3 Eq. (2):
  token loop of the GDN update from S0 (zero by default) over each tail, with
  the readout o_t = S_t (scale q_t).
  With ``scalar_decay``: the Mamba-2 family that the LinearKV page sets beside
  GDN (scalar per-token transition), S_t = alpha_t S_{t-1} + beta_t v_t k_t^T.
* :func:`chunk_operator` -- "LinearKV: One Cached State Suffices for
  Position-Independent Caching in Hybrid LLMs", composition passage: T_C as
  the product of the chunk's per-token transitions (latest on the left) and
  S_local as the state reached from an empty start.
* :func:`compose` -- same passage: the closed form
  S_K = T_{C_K}...T_{C_2} S_local_1 + ... + S_local_K, each carried product
  formed on its own.

State layout: S in R^{d_v x d_k}, row-major; T_C row-major d_k x d_k as the
pages' left operator on the transposed state (S_out = S_in T_C^T + S_local).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None


class _Dims(ctypes.Structure):
    _fields_ = [
        ("n_seqs", ctypes.c_int64),
        ("h_k", ctypes.c_int64),
        ("h_v", ctypes.c_int64),
        ("d_k", ctypes.c_int64),
        ("d_v", ctypes.c_int64),
        ("l2norm_qk", ctypes.c_int32),
        ("n_threads", ctypes.c_int32),
        ("scale", ctypes.c_double),
        ("scalar_decay", ctypes.c_int32),
    ]


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c into oracle/_build/libgdn_oracle.so (gcc, -O2)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _open(path: str):
    """Load a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER
    d = ctypes.c_void_p
    lib.gdn_oracle_replay.argtypes = [P(_Dims), d, d, d, d, d, d, d, d, d, d, ctypes.c_int64]
    lib.gdn_oracle_chunk_operator.argtypes = [P(_Dims), d, d, d, d, d, d, d]
    lib.gdn_oracle_compose.argtypes = [P(_Dims), ctypes.c_int64, d, d, d, d]
    lib.gdn_oracle_num_threads.argtypes = [ctypes.c_int32]
    for f in (lib.gdn_oracle_replay, lib.gdn_oracle_chunk_operator, lib.gdn_oracle_compose,
              lib.gdn_oracle_num_threads):
        f.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _open(build())
    return _lib


def _f64(x):
    return None if x is None else np.ascontiguousarray(x, dtype=np.float64)


def _ptr(x):
    return None if x is None else x.ctypes.data_as(ctypes.c_void_p)


def num_threads(requested: int = 0) -> int:
    """Threads the oracle uses for ``requested`` (0 = all online cores)."""
    return int(_load().gdn_oracle_num_threads(int(requested)))


def replay(q, k, v, g, beta, cu_seqlens, S0=None, *, l2norm_qk=True, scale=1.0, want_O=True,
           sel=None, n_threads=0, scalar_decay=False):
    """Token-loop replay.  Shapes: q,k [T,h_k,d_k]; v [T,h_v,d_v]; g,beta [T,h_v];
    cu_seqlens [n+1]; S0 [n,h_v,d_v,d_k] or None.  ``sel``: optional list of
    (sequence, v-head) pairs to compute (others stay zero).  ``scalar_decay``:
    the Mamba-2 family's scalar transition T_t = alpha_t I instead of GDN's.
    Returns (S, O) in fp64; O is None when ``want_O`` is False."""
    q, k, v, g, beta, S0 = map(_f64, (q, k, v, g, beta, S0))
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    T, h_k, d_k = k.shape
    h_v, d_v = v.shape[1], v.shape[2]
    n = cu.shape[0] - 1
    dims = _Dims(n, h_k, h_v, d_k, d_v, int(bool(l2norm_qk)), int(n_threads), float(scale), int(bool(scalar_decay)))
    S = np.zeros((n, h_v, d_v, d_k), dtype=np.float64)
    O = np.zeros((T, h_v, d_v), dtype=np.float64) if want_O else None
    sel_arr = None
    n_sel = 0
    if sel is not None:
        sel_arr = np.ascontiguousarray(np.asarray(sel, dtype=np.int64).reshape(-1, 2))
        n_sel = sel_arr.shape[0]
    rc = _load().gdn_oracle_replay(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                   _ptr(cu), _ptr(S0), _ptr(O), _ptr(S), _ptr(sel_arr), n_sel)
    if rc != 0:
        raise ValueError("gdn_oracle_replay: bad dims")
    return S, O


def chunk_operator(k, g, beta, v, cu_seqlens, *, h_k=None, l2norm_qk=True, n_threads=0, scalar_decay=False):
    """(T_C, S_local) per chunk (sequence of cu_seqlens) and v-head.
    Returns T [n,h_v,d_k,d_k] and S_local [n,h_v,d_v,d_k], fp64."""
    k, g, beta, v = map(_f64, (k, g, beta, v))
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    _, hk, d_k = k.shape
    h_v, d_v = v.shape[1], v.shape[2]
    n = cu.shape[0] - 1
    dims = _Dims(n, hk, h_v, d_k, d_v, int(bool(l2norm_qk)), int(n_threads), 1.0, int(bool(scalar_decay)))
    Tc = np.zeros((n, h_v, d_k, d_k), dtype=np.float64)
    Sl = np.zeros((n, h_v, d_v, d_k), dtype=np.float64)
    rc = _load().gdn_oracle_chunk_operator(ctypes.byref(dims), _ptr(k), _ptr(g), _ptr(beta), _ptr(v),
                                           _ptr(cu), _ptr(Tc), _ptr(Sl))
    if rc != 0:
        raise ValueError("gdn_oracle_chunk_operator: bad dims")
    return Tc, Sl


def compose(T, S_local, S_in=None, *, n_threads=0):
    """Closed-form composition.  T [K,h,d_k,d_k]; S_local [K,h,d_v,d_k];
    S_in [h,d_v,d_k] or None.  Returns S_K [h,d_v,d_k], fp64."""
    T, S_local, S_in = map(_f64, (T, S_local, S_in))
    K, h, d_k, _ = T.shape
    d_v = S_local.shape[2]
    dims = _Dims(1, h, h, d_k, d_v, 0, int(n_threads), 1.0, 0)
    out = np.zeros((h, d_v, d_k), dtype=np.float64)
    rc = _load().gdn_oracle_compose(ctypes.byref(dims), K, _ptr(T), _ptr(S_local), _ptr(S_in), _ptr(out))
    if rc != 0:
        raise ValueError("gdn_oracle_compose: bad dims")
    return out


def rel_err(x, ref) -> float:
    """Relative Frobenius error ||x - ref|| / ||ref|| over the whole tensor
    (absolute norm when ||ref|| is zero)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = float(np.linalg.norm((x - ref).ravel()))
    den = float(np.linalg.norm(ref.ravel()))
    return num / den if den > 0 else num
