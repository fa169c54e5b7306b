"""GB300-native Gated DeltaNet tail-replay state rebuild.

The computation lives in libgdn.so (CUDA for sm_103a, C ABI in include/gdn.h);
this package builds it (``build_lib``) and binds it (``api``: gdn_replay,
gdn_chunk_operator, gdn_compose, gdn_get_status, gdn_workspace_bytes).
"""
_API = ("gdn_replay", "gdn_replay_noalloc", "gdn_chunk_operator", "gdn_compose", "gdn_get_status", "gdn_workspace_bytes")


def __getattr__(name):
    if name in _API:
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
