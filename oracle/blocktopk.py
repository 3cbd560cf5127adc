"""Plain, slow CPU oracle of block top-k decode attention (numpy; test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this module.  It shares nothing with the CUDA path.

What the method computes, and where the pages say so:

* Block top-k attention ranks each key block by the mean of its key vectors and keeps
  only the k best blocks for each query group (Pith review of "Kinetics: Rethinking
  Test-Time Scaling Laws", section "What carries the argument").  The mean key of a block
  is its centroid; the query group is the set of query heads sharing one KV head (GQA).
* A block is one KV page of 16 tokens and k is counted in pages (Kinetics README,
  section "Benchmark Block TopK Attention throughput": ``--page_size 16 --topk_page 64``),
  and the benchmark is a paged decode of one decoder layer (same section).
* The selected blocks replace the quadratic KV term of the eFLOPs cost model with a
  term linear in the generated length (same Pith section, the C_TTS equation).

Readings taken where the pages are silent (each is listed with its reason in the
design notes of the repository):

1. Group aggregation: the block score is the SUM over the group's query heads of
   q_h . c_j.  (Sum and mean rank identically.)
2. The final block (the one holding the current token, possibly partial) is always
   kept and counts toward k; it is never scored.  If the row has nb <= k blocks,
   every block is kept.
3. Ties in score go to the lower block index.
4. The softmax scale sm_scale multiplies q . k inside the exponent; scoring ignores it
   (ranking is invariant to a positive scale).
5. Precision: scores, softmax and outputs are computed in float64 from float32
   centroids: keys are summed in float32 in ascending token order and scaled by 1/16
   (exact).  This fp32 centroid is what selection is judged against.  The library stores a
   bf16 cache's centroid as a pair of bf16 codes (``centroid_pair``: the fp32 mean rounded
   to bf16, and the rounding residual rounded to bf16); ``store="bf16"`` rounds the
   centroid to its first code, the value the library's block scores are computed from.
6. Acceptance of another implementation's selection: it may differ from this oracle's
   only on blocks whose oracle scores lie within 1e-3 (relative) of the last kept score;
   ``valid_selections`` lists every kept set that rule admits.

Parity pins for every function live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import itertools
import math
from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np

BLOCK = 16


# --------------------------------------------------------------------------------------
# Stored-code helpers
# --------------------------------------------------------------------------------------
def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); result stays float32.

    bfloat16 keeps the top 16 bits of the IEEE binary32 pattern.  Round-to-nearest-even
    adds half of the dropped range (0x7FFF) plus the parity of the kept least
    significant bit, then truncates.  NaNs stay NaN (quiet bit forced).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    keep_lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + keep_lsb) & np.uint64(0xFFFF0000)).astype(np.uint32)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = ((u[nan] | np.uint64(0x00400000)) & np.uint64(0xFFFF0000)).astype(np.uint32)
    return r.view(np.float32).reshape(x.shape)


def _store(x32: np.ndarray, store: str) -> np.ndarray:
    if store == "bf16":
        return round_to_bf16(x32)
    if store == "f32":
        return x32.astype(np.float32)
    raise ValueError(store)


# --------------------------------------------------------------------------------------
# Step 1: block centroid (mean key vector)
# --------------------------------------------------------------------------------------
def block_centroid(keys: np.ndarray, store: str = "f32") -> np.ndarray:
    """Mean of one block's 16 key vectors.

    Blocks are ranked by the mean of their keys (Pith review, "What carries the
    argument").  keys: [16, d] float32 values of one (page, KV head).  Summed in float32
    in ascending token order, multiplied by 1/16 (a power of two, so exact), rounded to
    the storage type.
    """
    keys = np.asarray(keys, dtype=np.float32)
    assert keys.shape[0] == BLOCK
    acc = keys[0].copy()
    for t in range(1, BLOCK):
        acc = (acc + keys[t]).astype(np.float32)
    mean = (acc * np.float32(1.0 / BLOCK)).astype(np.float32)
    return _store(mean, store)


def centroids(k_pages: np.ndarray, page_ids: Sequence[int], store: str) -> np.ndarray:
    """Centroids of the listed physical pages for every KV head.

    k_pages: [P, H, 16, d] float32; returns [len(page_ids), H, d] float32 holding the
    stored (bf16 or fp32) values.  Same arithmetic as ``block_centroid``, applied to
    all heads of a page at once (elementwise, still ascending token order).
    """
    ids = np.asarray(page_ids, dtype=np.int64)
    blk = np.asarray(k_pages[ids], dtype=np.float32)          # [n, H, 16, d]
    acc = blk[:, :, 0, :].copy()
    for t in range(1, BLOCK):
        acc = (acc + blk[:, :, t, :]).astype(np.float32)
    mean = (acc * np.float32(1.0 / BLOCK)).astype(np.float32)
    return _store(mean, store)


def centroid_pair(k_pages: np.ndarray, page_ids: Sequence[int]) -> Tuple[np.ndarray, np.ndarray]:
    """The two bf16 codes a bf16 cache stores for each listed page's centroid.

    hi = the fp32 mean rounded to bf16 (round-to-nearest-even); lo = (mean - hi) rounded
    to bf16.  The fp32 difference is exact (hi is the rounding of the mean, so the two lie
    within a factor of two of each other), hence hi + lo equals the fp32 mean to about 2^-16
    of its size.  Returns (hi, lo), each [len(page_ids), H, d] float32 holding bf16 values.
    """
    c32 = centroids(k_pages, page_ids, "f32")
    hi = round_to_bf16(c32)
    lo = round_to_bf16((c32 - hi).astype(np.float32))
    return hi, lo


# --------------------------------------------------------------------------------------
# Step 2: group score of each candidate block
# --------------------------------------------------------------------------------------
def group_scores(q_group: np.ndarray, cents: np.ndarray) -> np.ndarray:
    """s_j = sum over the group's query heads g of (q_g . c_j), in float64.

    Selection happens once per GQA query group (Pith review, "What carries the
    argument"), so there is one score per block for the whole group; the aggregation over the
    group is a sum (reading 1).  q_group: [G, d]; cents: [n, d]; returns [n].
    """
    q = np.asarray(q_group, dtype=np.float64)
    c = np.asarray(cents, dtype=np.float64)
    s = np.zeros(c.shape[0], dtype=np.float64)
    for g in range(q.shape[0]):
        s += (c * q[g][None, :]).sum(axis=1)
    return s


# --------------------------------------------------------------------------------------
# Step 3: top-k block selection
# --------------------------------------------------------------------------------------
def select_blocks(scores: Sequence[float], nb: int, k: int) -> List[int]:
    """Logical block ids kept for one (sequence, KV head) row, ascending.

    the k best blocks per query group (Pith review, "What carries the argument"); k counted in
    pages (Kinetics README, "Benchmark Block TopK Attention throughput").  The final
    block nb-1 is always kept and counts toward k (reading 2); the other k-1 are the
    highest-scoring of blocks 0..nb-2, ties to the lower index (reading 3).  With
    nb <= k every block is kept.  ``scores`` holds s_j for j = 0..nb-2.
    """
    if nb <= 0:
        return []
    if nb <= k:
        return list(range(nb))
    assert len(scores) >= nb - 1
    order = sorted(range(nb - 1), key=lambda j: (-float(scores[j]), j))
    chosen = order[: k - 1]
    return sorted(chosen + [nb - 1])


def valid_selections(scores: Sequence[float], nb: int, k: int, rel: float = 1e-3,
                     limit: int = 100000) -> List[List[int]]:
    """Every kept list an implementation may return for one row under the acceptance rule.

    The rule: a kept set may differ from ``select_blocks``'s only on blocks whose scores lie
    within ``rel`` (relative) of the last kept score s_(k), i.e. where the oracle's k-th and
    (k+1)-th scores nearly tie.  So the blocks kept outside that band are kept by every
    admissible set, and the rest of the k-1 scored places go to any choice of blocks inside
    the band.  Returns the sets ascending (the oracle's own among them); raises when there
    are more than ``limit``.
    """
    base = select_blocks(scores, nb, k)
    if nb <= k:
        return [base]
    m = k - 1
    if m == 0:
        return [base]
    cand = [float(scores[j]) for j in range(nb - 1)]
    order = sorted(range(nb - 1), key=lambda j: (-cand[j], j))
    t = cand[order[m - 1]]
    band = rel * abs(t)
    near = [j for j in range(nb - 1) if abs(cand[j] - t) <= band]
    near_set = set(near)
    core = [j for j in base[:-1] if j not in near_set]
    r = m - len(core)
    n_sets = math.comb(len(near), r)
    if n_sets > limit:
        raise ValueError(f"{n_sets} admissible selections (limit {limit})")
    return [sorted(core + list(c) + [nb - 1]) for c in itertools.combinations(near, r)]


# --------------------------------------------------------------------------------------
# Step 4: softmax attention over the kept tokens
# --------------------------------------------------------------------------------------
def attend(q_group: np.ndarray, keys: np.ndarray, vals: np.ndarray,
           sm_scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """Softmax attention of each query head over the given tokens, float64.

    z_t = sm_scale * q . k_t;  o = sum_t softmax(z)_t v_t;  lse = log sum_t exp(z_t).
    The paged decode of one layer (Kinetics README, "Benchmark Block TopK Attention
    throughput") restricted to the kept blocks.  Returns out [G, d] and lse [G].
    """
    q = np.asarray(q_group, dtype=np.float64)
    kk = np.asarray(keys, dtype=np.float64)
    vv = np.asarray(vals, dtype=np.float64)
    z = sm_scale * (q @ kk.T)                   # [G, T]
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    den = e.sum(axis=1)
    out = (e @ vv) / den[:, None]
    lse = m[:, 0] + np.log(den)
    return out, lse


def row_tokens(k_pages: np.ndarray, v_pages: np.ndarray, table_row: Sequence[int],
               seq_len: int, blocks: Iterable[int], h: int) -> Tuple[np.ndarray, np.ndarray]:
    """Gather the valid tokens (position < seq_len) of the given logical blocks."""
    ks, vs = [], []
    for j in blocks:
        p = int(table_row[j])
        n = min(BLOCK, seq_len - BLOCK * j)
        ks.append(np.asarray(k_pages[p, h, :n], dtype=np.float64))
        vs.append(np.asarray(v_pages[p, h, :n], dtype=np.float64))
    return np.concatenate(ks, axis=0), np.concatenate(vs, axis=0)


# --------------------------------------------------------------------------------------
# Whole decode step
# --------------------------------------------------------------------------------------
def decode_rows(q: np.ndarray, k_pages: np.ndarray, v_pages: np.ndarray,
                block_table: np.ndarray, seq_lens: np.ndarray, sm_scale: float,
                top_k: Optional[int], store: str,
                rows: Optional[Iterable[Tuple[int, int]]] = None) -> dict:
    """One decode step for the listed (sequence, KV head) rows (all rows by default).

    top_k=None gives dense decode (every block kept).  Inputs are the host arrays of
    the workload (float32 values of the stored dtype); q: [B, Hq, d]; k/v_pages:
    [P, H, 16, d]; block_table: [B, max_blocks]; seq_lens: [B].  ``store`` is the
    centroid storage type.  Rows not computed are left NaN / -1.
    """
    B, Hq, d = q.shape
    H = k_pages.shape[1]
    G = Hq // H
    maxb = block_table.shape[1]
    kdim = top_k if top_k is not None else maxb
    out = np.full((B, Hq, d), np.nan)
    lse = np.full((B, Hq), np.nan)
    sel = np.full((B, H, kdim), -1, dtype=np.int64)
    scores = np.full((B, H, maxb), np.nan)
    if rows is None:
        rows = [(b, h) for b in range(B) for h in range(H)]
    cent_cache = {}
    for b, h in rows:
        L = int(seq_lens[b])
        nb = (L + BLOCK - 1) // BLOCK
        qg = q[b, h * G:(h + 1) * G]
        if top_k is None or nb <= top_k:
            blocks = list(range(nb))
        else:
            cand = [int(block_table[b, j]) for j in range(nb - 1)]
            need = [p for p in set(cand) if (p, h) not in cent_cache]
            if need:
                c = centroids(k_pages[:, h:h + 1], need, store)[:, 0]
                for p, cv in zip(need, c):
                    cent_cache[(p, h)] = cv
            cm = np.stack([cent_cache[(p, h)] for p in cand])
            s = group_scores(qg, cm)
            scores[b, h, :nb - 1] = s
            blocks = select_blocks(s, nb, top_k)
        sel[b, h, :len(blocks)] = blocks
        kk, vv = row_tokens(k_pages, v_pages, block_table[b], L, blocks, h)
        o, ls = attend(qg, kk, vv, sm_scale)
        out[b, h * G:(h + 1) * G] = o
        lse[b, h * G:(h + 1) * G] = ls
    return dict(out=out, lse=lse, sel=sel, scores=scores)


def blocktopk_decode(q, k_pages, v_pages, block_table, seq_lens, sm_scale, top_k,
                     store="f32", rows=None) -> dict:
    """Block top-k decode (score, select, attend) for the listed rows.

    store="f32" (fp32 centroids) is the reference selection; store="bf16" scores with the
    centroids rounded to bf16, the block scores a bf16 cache's first centroid code gives."""
    return decode_rows(q, k_pages, v_pages, block_table, seq_lens, sm_scale, top_k,
                       store, rows)


def dense_decode(q, k_pages, v_pages, block_table, seq_lens, sm_scale, rows=None) -> dict:
    """Dense paged decode over every block (the comparison baseline)."""
    return decode_rows(q, k_pages, v_pages, block_table, seq_lens, sm_scale, None,
                       "f32", rows)


# --------------------------------------------------------------------------------------
# Byte accounting (the algorithmic bytes a decode step must move)
# --------------------------------------------------------------------------------------
def sparse_kv_tokens(seq_len: int, top_k: Optional[int]) -> int:
    """Tokens whose K and V a row reads in one step: all of the kept blocks' valid ones."""
    nb = (seq_len + BLOCK - 1) // BLOCK
    if top_k is None or nb <= top_k:
        return seq_len
    return (top_k - 1) * BLOCK + (seq_len - BLOCK * (nb - 1))


def dense_kv_bytes_per_step(seq_len: int, num_kv_heads: int, head_dim: int,
                            esize: int) -> int:
    """K+V bytes dense decode reads for one sequence in one layer at context seq_len."""
    return 2 * seq_len * num_kv_heads * head_dim * esize


def decode_bytes(seq_lens: Sequence[int], num_kv_heads: int, group: int, head_dim: int,
                 top_k: Optional[int], esize: int) -> dict:
    """Algorithmic bytes of one decode step: kept K/V + scored centroids + Q and O.

    The K/V term is the per-step form of the cost model's KV-access term (Pith review,
    "What carries the argument": the quadratic term for dense attention, replaced by one
    linear in the generated length for block top-k).  Centroids are read only for
    scored blocks (rows with more than k blocks); Q and O are read / written once.
    """
    kv = cent = 0
    for L in seq_lens:
        L = int(L)
        nb = (L + BLOCK - 1) // BLOCK
        kv += 2 * sparse_kv_tokens(L, top_k) * num_kv_heads * head_dim * esize
        if top_k is not None and nb > top_k:
            cent += (nb - 1) * num_kv_heads * head_dim * esize
    qo = 2 * len(seq_lens) * num_kv_heads * group * head_dim * esize
    return dict(kv=kv, centroids=cent, qo=qo, total=kv + cent + qo)
