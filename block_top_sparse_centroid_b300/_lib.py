"""ctypes view of libkin.so (the C ABI declared in include/kin.h).

Loading fails loudly when the library has not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

from ctypes import POINTER, c_char_p, c_float, c_int, c_int32, c_int64, c_size_t, c_void_p

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkin.so")

KIN_OK = 0
KIN_ERR_INVALID_ARG = 1
KIN_ERR_UNSUPPORTED = 2
KIN_ERR_WORKSPACE = 3
KIN_ERR_CUDA = 4

KIN_F32 = 0
KIN_BF16 = 1

KIN_DEVERR_PAGE_ID = 1
KIN_DEVERR_SEQ_LEN = 2
KIN_DEVERR_TIMEOUT = 4

KIN_DECODE_APPEND_FINAL = 1

MODE_BLOCKTOPK = 0
MODE_DENSE = 1
MODE_TOKENTOPK = 2


class KvCache(ctypes.Structure):
    """Mirror of kin_kv_cache."""
    _fields_ = [("dtype", c_int), ("num_kv_heads", c_int32), ("head_dim", c_int32),
                ("page_size", c_int32), ("num_pages", c_int64), ("k_pages", c_void_p),
                ("v_pages", c_void_p)]


class DecodeArgs(ctypes.Structure):
    """Mirror of kin_decode_args."""
    _fields_ = [("batch", c_int32), ("num_q_heads", c_int32), ("max_blocks", c_int32),
                ("top_k", c_int32), ("sm_scale", c_float), ("q", c_void_p),
                ("block_table", c_void_p), ("seq_lens", c_void_p), ("centroids", c_void_p),
                ("out", c_void_p), ("lse", c_void_p), ("sel_blocks", c_void_p),
                ("scores", c_void_p), ("workspace", c_void_p), ("workspace_bytes", c_size_t),
                ("err_flag", c_void_p), ("flags", c_int32), ("shared_prefix_blocks", c_int32)]


# Every function include/kin.h declares, with its ctypes signature.
SIGNATURES = {
    "kin_status_str": (c_char_p, [c_int]),
    "kin_last_error": (c_char_p, []),
    "kin_workspace_size": (c_int, [POINTER(KvCache), POINTER(DecodeArgs), c_int32,
                                   POINTER(c_size_t)]),
    "kin_centroids_build": (c_int, [POINTER(KvCache), c_void_p, c_int64, c_void_p, c_void_p,
                                    c_void_p]),
    "kin_centroids_append": (c_int, [POINTER(KvCache), c_void_p, c_int32, c_void_p, c_void_p,
                                     c_void_p]),
    "kin_blocktopk_decode": (c_int, [POINTER(KvCache), POINTER(DecodeArgs), c_void_p]),
    "kin_dense_decode": (c_int, [POINTER(KvCache), POINTER(DecodeArgs), c_void_p]),
    "kin_token_topk_decode": (c_int, [POINTER(KvCache), POINTER(DecodeArgs), c_void_p]),
    "kin_blocktopk_decode_static": (c_int, [POINTER(KvCache), POINTER(DecodeArgs), c_void_p]),
    "kin_decode_timed": (c_int, [POINTER(KvCache), POINTER(DecodeArgs), c_int32,
                                 POINTER(c_void_p), c_void_p]),
}

_lib = None


def open_library(path: str) -> ctypes.CDLL:
    """A libkin build at `path` with every declared signature set (not cached)."""
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -m block_top_sparse_centroid_b300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load() -> ctypes.CDLL:
    """Load libkin.so once; raise if it is missing (build it with the package's build)."""
    global _lib
    if _lib is None:
        _lib = open_library(LIB_PATH)
    return _lib


class KinError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        name = lib.kin_status_str(status).decode()
        msg = lib.kin_last_error().decode()
        super().__init__(f"{where}: {name}: {msg}")
        self.status = status


def check(status: int, where: str) -> None:
    if status != KIN_OK:
        raise KinError(status, where)
