"""ctypes view of libgdn.so (declarations mirror include/gdn.h)."""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import build_lib

GDN_OK = 0
GDN_ERR_ARG = -1
GDN_ERR_SHAPE = -2
GDN_ERR_ALIGN = -3
GDN_ERR_UNSUPPORTED = -4
GDN_ERR_CUDA = -5
GDN_ERR_TIMEOUT = -6
GDN_ERR_NOMEM = -7

GDN_F32 = 0
GDN_BF16 = 1

GDN_QK_L2NORM = 1
GDN_STATE_ONLY = 2
GDN_PRECISE = 4
GDN_SCALAR_DECAY = 8

ERROR_NAMES = {
    GDN_ERR_ARG: "GDN_ERR_ARG", GDN_ERR_SHAPE: "GDN_ERR_SHAPE", GDN_ERR_ALIGN: "GDN_ERR_ALIGN",
    GDN_ERR_UNSUPPORTED: "GDN_ERR_UNSUPPORTED", GDN_ERR_CUDA: "GDN_ERR_CUDA",
    GDN_ERR_TIMEOUT: "GDN_ERR_TIMEOUT", GDN_ERR_NOMEM: "GDN_ERR_NOMEM",
}


class GdnDims(ctypes.Structure):
    _fields_ = [
        ("n_seqs", ctypes.c_int32),
        ("total_tokens", ctypes.c_int32),
        ("h_k", ctypes.c_int32),
        ("h_v", ctypes.c_int32),
        ("d_k", ctypes.c_int32),
        ("d_v", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("flags", ctypes.c_uint32),
        ("scale", ctypes.c_float),
    ]


class GdnError(RuntimeError):
    def __init__(self, code: int, where: str, message: str):
        self.code = code
        super().__init__(f"{where} failed: {ERROR_NAMES.get(code, code)}: {message}")


_lock = threading.Lock()
_lib = None
_VP = ctypes.c_void_p
_PD = ctypes.POINTER(GdnDims)

SIGNATURES = {
    "gdn_replay": ([_PD, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP], ctypes.c_int),
    "gdn_replay_noalloc": ([_PD, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP], ctypes.c_int),
    "gdn_chunk_operator": ([_PD, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP], ctypes.c_int),
    "gdn_compose": ([_PD, ctypes.c_int32, _VP, _VP, _VP, _VP, _VP], ctypes.c_int),
    "gdn_get_status": ([_VP], ctypes.c_int),
    "gdn_last_error": ([], ctypes.c_char_p),
    "gdn_workspace_bytes": ([_PD], ctypes.c_size_t),
    "gdn_abi_version": ([], ctypes.c_int),
    "gdn_set_stage_event": ([_VP], None),
    "gdn_set_wait_limit_ns": ([ctypes.c_uint64], None),
}


def header_functions() -> list[str]:
    """Names of the functions that include/*.h declare."""
    names = []
    for h in sorted(os.listdir(build_lib.INCLUDE)):
        if h.endswith(".h"):
            text = open(os.path.join(build_lib.INCLUDE, h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w ]*?[\s*]+(gdn_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def load(build: bool = False):
    """Load libgdn.so.  With ``build=True`` compile it first when missing or stale.
    Raises RuntimeError when the library is absent: there is no fallback."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build:
            build_lib.build_library()
        if not os.path.exists(build_lib.LIB_PATH):
            raise RuntimeError(
                f"{build_lib.LIB_PATH} is missing: build it with "
                "`python -m gated_deltanet_state_chunked_gb300.build_lib` (needs nvcc)")
        lib = ctypes.CDLL(build_lib.LIB_PATH)
        for name, (args, res) in SIGNATURES.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
    return _lib


def check(rc: int, where: str) -> None:
    if rc != GDN_OK:
        msg = _lib.gdn_last_error().decode() if _lib is not None else ""
        raise GdnError(rc, where, msg)
