"""Block top-k (centroid-scored) sparse decode attention for B300 (sm_103a).

The compute runs in libkin.so (hand-written CUDA behind a C ABI, include/kin.h); this
package is its thin Python binding.  Every call loads the library on first use and
raises if it has not been built (``python -m block_top_sparse_centroid_b300.build``):
there is no CPU or eager fallback.
"""
from . import _lib
from ._lib import KinError, load as load_library
from .api import (BLOCK, PagedKVCache, PreparedDecode, Workspace, blocktopk_decode,
                  centroids_append, centroids_build, decode_timed, dense_decode,
                  prepare_blocktopk_decode, prepare_dense_decode, prepare_token_topk_decode,
                  token_topk_decode, workspace_size)

__all__ = ["BLOCK", "KinError", "PagedKVCache", "PreparedDecode", "Workspace",
           "blocktopk_decode", "centroids_append", "centroids_build", "decode_timed",
           "dense_decode", "prepare_blocktopk_decode", "prepare_dense_decode",
           "prepare_token_topk_decode", "token_topk_decode", "workspace_size", "load_library"]
