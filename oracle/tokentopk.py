"""Plain, slow CPU oracle of token-level ("oracle") top-k decode attention (numpy; test
infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this module.  It shares nothing with the CUDA path.

What it computes, and where the pages say so:

* Oracle top-k attention is sparse attention whose kept keys are the ones with the largest
  exact scores q . k -- a perfect selection, used as the accuracy upper bound that block
  top-k approaches (scime summary of "Kinetics: Rethinking Test-Time Scaling Laws", "Key
  results"; Pith review of the same paper, the "assumptions" list, where oracle top-k is
  the perfect-selection proxy; the codewithpapers entry of the paper lists a
  ``topk_sparsity`` function in the official repository's attention utilities).
* Block top-k, its deployable approximation, ranks 16-token pages by their mean key per
  query group (Pith review, "What carries the argument"); oracle top-k ranks single
  tokens by their exact scores.

Readings taken where the pages are silent (each is listed with its reason in the design
notes of the repository):

T1. Granularity: one selection per (sequence, KV head) row, scoring token t by the SUM over
    the group's query heads of q_g . k_t -- the query-group aggregation of block top-k
    (its reading 1), so that both methods choose the K/V a group reads once.
T2. Budget: ``top_tokens`` = B tokens per row; the equal-KV budget of block top-k with k
    pages is B = 16 k.  A row of L <= B tokens keeps every token.
T3. No token is forced in: the current token competes like every other one.
T4. Ties in score go to the lower token position.
T5. Precision: scores in float64 from the stored key values; attention as ``attend``.
T6. Acceptance of another implementation's kept set: it may differ from this oracle's only
    on tokens whose oracle scores lie within ``tol`` of the B-th largest oracle score
    (``token_admissible``).

Parity pins live in ``tests/test_oracle_token_pins.py``.
"""
from __future__ import annotations

from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np

from .blocktopk import BLOCK, attend, row_tokens


def token_scores(q_group: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """s_t = sum over the group's query heads g of (q_g . k_t), float64 (reading T1).

    q_group: [G, d]; keys: [T, d]; returns [T]."""
    q = np.asarray(q_group, dtype=np.float64)
    k = np.asarray(keys, dtype=np.float64)
    s = np.zeros(k.shape[0], dtype=np.float64)
    for g in range(q.shape[0]):
        s += (k * q[g][None, :]).sum(axis=1)
    return s


def select_tokens(scores: Sequence[float], budget: int) -> List[int]:
    """Token positions kept for one row, ascending: the ``budget`` highest scores, ties to
    the lower position (readings T2-T4); every position when the row is not longer."""
    n = len(scores)
    if n <= budget:
        return list(range(n))
    order = sorted(range(n), key=lambda t: (-float(scores[t]), t))
    return sorted(order[:budget])


def token_admissible(scores: Sequence[float], kept: Sequence[int], budget: int,
                     tol: float) -> bool:
    """Whether ``kept`` is a kept set the acceptance rule (reading T6) admits: the right
    number of distinct positions of the row, differing from ``select_tokens``'s only on
    tokens whose scores lie within ``tol`` of the oracle's B-th largest score."""
    n = len(scores)
    ref = select_tokens(scores, budget)
    kept = [int(t) for t in kept]
    if len(set(kept)) != len(kept) or len(kept) != len(ref):
        return False
    if any(t < 0 or t >= n for t in kept):
        return False
    if n <= budget:
        return sorted(kept) == ref
    sb = sorted((float(s) for s in scores), reverse=True)[budget - 1]
    ks, rs = set(kept), set(ref)
    return (all(float(scores[t]) >= sb - tol for t in ks - rs) and
            all(float(scores[t]) <= sb + tol for t in rs - ks))


def row_keys_values(k_pages: np.ndarray, v_pages: np.ndarray, table_row: Sequence[int],
                    seq_len: int, h: int) -> Tuple[np.ndarray, np.ndarray]:
    """Every token of one row in position order: keys, values [L, d] float64."""
    nb = (seq_len + BLOCK - 1) // BLOCK
    return row_tokens(k_pages, v_pages, table_row, seq_len, range(nb), h)


def tokentopk_rows(q: np.ndarray, k_pages: np.ndarray, v_pages: np.ndarray,
                   block_table: np.ndarray, seq_lens: np.ndarray, sm_scale: float,
                   top_tokens: int, rows: Optional[Iterable[Tuple[int, int]]] = None) -> dict:
    """One token top-k decode step for the listed (sequence, KV head) rows (all by default).

    Same inputs as ``blocktopk.decode_rows``.  Returns out [B, Hq, d], lse [B, Hq], sel
    [B, H, top_tokens] (kept positions ascending, -1 padded) and scores [B, H, 16 max_blocks]
    (NaN where not computed)."""
    B, Hq, d = q.shape
    H = k_pages.shape[1]
    G = Hq // H
    maxb = block_table.shape[1]
    out = np.full((B, Hq, d), np.nan)
    lse = np.full((B, Hq), np.nan)
    sel = np.full((B, H, top_tokens), -1, dtype=np.int64)
    scores = np.full((B, H, maxb * BLOCK), np.nan)
    if rows is None:
        rows = [(b, h) for b in range(B) for h in range(H)]
    for b, h in rows:
        L = int(seq_lens[b])
        qg = q[b, h * G:(h + 1) * G]
        kk, vv = row_keys_values(k_pages, v_pages, block_table[b], L, h)
        s = token_scores(qg, kk)
        scores[b, h, :L] = s
        kept = select_tokens(s, top_tokens)
        sel[b, h, :len(kept)] = kept
        o, ls = attend(qg, kk[kept], vv[kept], sm_scale)
        out[b, h * G:(h + 1) * G] = o
        lse[b, h * G:(h + 1) * G] = ls
    return dict(out=out, lse=lse, sel=sel, scores=scores)


def tokentopk_decode(q, k_pages, v_pages, block_table, seq_lens, sm_scale, top_tokens,
                     rows=None) -> dict:
    """Token-level top-k decode (score every token, keep the top ``top_tokens``, attend)."""
    return tokentopk_rows(q, k_pages, v_pages, block_table, seq_lens, sm_scale, top_tokens,
                          rows)


def token_decode_bytes(seq_lens: Sequence[int], num_kv_heads: int, group: int, head_dim: int,
                       top_tokens: int, esize: int) -> dict:
    """Algorithmic bytes of one token top-k step: every key of every row read once (the
    scoring), the kept tokens' keys and values read once more (the attention), and the
    queries and outputs.  Scores and kept lists are workspace, counted separately."""
    H, G, d = num_kv_heads, group, head_dim
    all_k = sum(int(L) for L in seq_lens) * H * d * esize
    kept = sum(min(int(L), top_tokens) for L in seq_lens) * H * 2 * d * esize
    qo = 2 * len(seq_lens) * H * G * d * esize
    return {"all_k": all_k, "kept_kv": kept, "qo": qo, "total": all_k + kept + qo}
