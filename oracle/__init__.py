"""CPU oracle for block top-k (centroid-scored) decode attention.

TEST INFRASTRUCTURE, not part of the product.  Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import or run it.  It
shares no code with the CUDA library: it reads the same seeded host inputs and nothing
else, and it never reads anything the CUDA path computed.

See ``oracle.blocktopk`` (block top-k) and ``oracle.tokentopk`` (token-level top-k) for
the methods and the passages each function follows.
"""
from .blocktopk import (BLOCK, round_to_bf16, block_centroid, centroids, centroid_pair,
                        group_scores, valid_selections,
                        select_blocks, attend, row_tokens, decode_rows, blocktopk_decode,
                        dense_decode, decode_bytes, dense_kv_bytes_per_step,
                        sparse_kv_tokens)
from .tokentopk import (token_scores, select_tokens, token_admissible, row_keys_values,
                        tokentopk_rows, tokentopk_decode, token_decode_bytes)

__all__ = ["BLOCK", "round_to_bf16", "block_centroid", "centroids", "centroid_pair",
           "valid_selections", "group_scores",
           "select_blocks", "attend", "row_tokens", "decode_rows", "blocktopk_decode",
           "dense_decode", "decode_bytes", "dense_kv_bytes_per_step", "sparse_kv_tokens",
           "token_scores", "select_tokens", "token_admissible", "row_keys_values",
           "tokentopk_rows", "tokentopk_decode", "token_decode_bytes"]
