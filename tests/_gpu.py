"""Helpers for the GPU parity tests: upload seeded inputs, run the library through its
C ABI binding, and compare with the CPU oracle row by row.

Tolerances:
* bf16 outputs: max-abs 2e-2 and mean-abs 2e-3 per row (the acceptance bar of the
  method's specification); lse within 2e-3 (the kernel rounds each softmax weight to
  bf16 before summing it, a relative error of at most 2^-9 in the sum, i.e. 2e-3 in ln).
* fp32 outputs: max-abs 1e-4, lse 1e-5 (fp32 accumulation and exp2 over <= 2^14 terms).
* Centroids: bit-exact (both sides sum the 16 keys in fp32 in token order; bf16 caches
  store the mean and its residual, each rounded to bf16 the same way).
* Scores: the library's block scores come from the first bf16 centroid code, so they are
  compared with the oracle's scores of bf16-rounded centroids:
  |s_gpu - s_oracle| <= 2e-5 * sum_{g,i} |q_gi c_i| (fp32 dot products of <= 2048 terms
  against an fp64 reference).
* Selection: judged against the oracle's selection with fp32 centroids.  Bit-exact, except
  where the oracle's last kept and first dropped scores differ by less than 1e-3
  relative: then the kept set must be one of the sets that rule admits
  (oracle.valid_selections), and the row's output and lse are compared with the
  oracle's attention over that admissible set.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle as O
import workloads as W
import block_top_sparse_centroid_b300 as K

OUT_MAX_ABS = {"bf16": 2e-2, "f32": 1e-4}
OUT_MEAN_ABS = {"bf16": 2e-3, "f32": 2e-5}
LSE_ABS = {"bf16": 2e-3, "f32": 1e-5}
SCORE_REL = 2e-5
TIE_REL = 1e-3


def device():
    return torch.device("cuda:0")


class DeviceState:
    """Device copies of a workload plus its centroid table built by the library."""

    def __init__(self, inp: W.Inputs, dev=None, build=True, append=True):
        dev = dev or device()
        self.inp = inp
        self.dev = dev
        self.cache = K.PagedKVCache(inp.k_pages.to(dev), inp.v_pages.to(dev))
        self.q = inp.q.to(dev)
        self.table = inp.block_table.to(dev)
        self.lens = inp.seq_lens.to(dev)
        cfg = inp.cfg
        self.cents = torch.zeros(self.cache.centroid_shape, dtype=W.torch_dtype(cfg.dtype),
                                 device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        if build:
            # pages completed before this step (prefill), then the pages the current token
            # just completed (one append step)
            full = set(inp.complete_pages().tolist())
            last = inp.last_pages().tolist()
            just = sorted({p for b, p in enumerate(last)
                           if int(inp.seq_lens[b]) % W.BLOCK == 0} & full)
            before = sorted(full - set(just))
            if before:
                K.centroids_build(self.cache, self.cents,
                                  page_ids=torch.tensor(before, dtype=torch.int32, device=dev),
                                  err_flag=self.err)
            self.just_pages = just
            if just and append:
                K.centroids_append(self.cache, torch.tensor(just, dtype=torch.int32, device=dev),
                                   self.cents, err_flag=self.err)

    def refresh_q(self):
        self.q = self.inp.q.to(self.dev)

    def decode(self, dense=False, append_final=False, shared_prefix_blocks=0):
        cfg = self.inp.cfg
        B, Hq, H = cfg.batch, cfg.num_q_heads, cfg.num_kv_heads
        out = torch.full((B, Hq, cfg.head_dim), float("nan"), dtype=self.q.dtype, device=self.dev)
        lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=self.dev)
        if dense:
            K.dense_decode(self.cache, self.q, self.table, self.lens, cfg.sm_scale, out=out,
                           lse=lse, err_flag=self.err, centroids=self.cents,
                           append_final=append_final, shared_prefix_blocks=shared_prefix_blocks)
            torch.cuda.synchronize()
            return dict(out=out.float().cpu().numpy(), lse=lse.cpu().numpy())
        sel = torch.full((B, H, cfg.top_k), -7, dtype=torch.int32, device=self.dev)
        scores = torch.full((B, H, self.inp.max_blocks), float("nan"), dtype=torch.float32,
                            device=self.dev)
        K.blocktopk_decode(self.cache, self.q, self.table, self.lens, self.cents, cfg.top_k,
                           cfg.sm_scale, out=out, lse=lse, sel_blocks=sel, scores=scores,
                           err_flag=self.err, append_final=append_final,
                           shared_prefix_blocks=shared_prefix_blocks)
        torch.cuda.synchronize()
        return dict(out=out.float().cpu().numpy(), lse=lse.cpu().numpy(),
                    sel=sel.cpu().numpy(), scores=scores.cpu().numpy())

    def token_decode(self, budget: int, events=None):
        """One token-level top-k decode (kin_token_topk_decode) of the current state."""
        cfg = self.inp.cfg
        B, Hq, H = cfg.batch, cfg.num_q_heads, cfg.num_kv_heads
        out = torch.full((B, Hq, cfg.head_dim), float("nan"), dtype=self.q.dtype, device=self.dev)
        lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=self.dev)
        sel = torch.full((B, H, budget), -7, dtype=torch.int32, device=self.dev)
        scores = torch.full((B, H, 16 * self.inp.max_blocks), float("nan"), dtype=torch.float32,
                            device=self.dev)
        K.token_topk_decode(self.cache, self.q, self.table, self.lens, budget, cfg.sm_scale,
                            out=out, lse=lse, sel_tokens=sel, scores=scores, err_flag=self.err,
                            events=events)
        torch.cuda.synchronize()
        return dict(out=out.float().cpu().numpy(), lse=lse.cpu().numpy(), sel=sel.cpu().numpy(),
                    scores=scores.cpu().numpy())

    def error_bits(self) -> int:
        torch.cuda.synchronize()
        return int(self.err.item())


def oracle_row(inp: W.Inputs, b: int, h: int, dense: bool) -> dict:
    """The oracle's result for one row: fp32 centroids (the reference selection)."""
    cfg = inp.cfg
    rp = W.row_problem(inp, b, h)
    if dense:
        return O.dense_decode(rp["q"], rp["k_pages"], rp["v_pages"], rp["block_table"],
                              rp["seq_lens"], cfg.sm_scale)
    return O.blocktopk_decode(rp["q"], rp["k_pages"], rp["v_pages"], rp["block_table"],
                              rp["seq_lens"], cfg.sm_scale, cfg.top_k, store="f32")


def admissible_set(sel_g, scores_o, nb, k):
    """The admissible kept set (oracle.valid_selections over the oracle's scores) equal to
    the GPU's kept list; fails when the GPU's list is not one of them."""
    g = [int(x) for x in sel_g if x >= 0]
    assert len(g) == min(nb, k) and g == sorted(set(g)) and g[-1] == nb - 1, (g, nb, k)
    if g == O.select_blocks(list(np.asarray(scores_o[: max(nb - 1, 0)], np.float64)), nb, k):
        return g
    sets = O.valid_selections(list(np.asarray(scores_o[: max(nb - 1, 0)], np.float64)), nb, k,
                              rel=TIE_REL)
    for cand in sets:
        if cand == g:
            return cand
    raise AssertionError(f"kept list {g} is not admissible (oracle: {sets[:3]} ...)")


def compare_rows(inp: W.Inputs, res: dict, rows, dense=False, q_host=None) -> dict:
    """Compare the GPU result of the listed rows with the oracle; returns statistics:
    rows checked, near_tie_rows (kept set admissible but not the oracle's own; output
    checked against the oracle over that set), bf16_rank_diff (rows whose kept set differs
    from the ranking by bf16-rounded centroids, i.e. where the residual plane mattered)."""
    cfg = inp.cfg
    G = cfg.group
    dt = cfg.dtype
    stats = dict(rows=0, near_tie_rows=0, bf16_rank_diff=0, max_abs=0.0, max_lse=0.0)
    for b, h in rows:
        ref = oracle_row(inp, b, h, dense)
        L = int(inp.seq_lens[b])
        nb = (L + W.BLOCK - 1) // W.BLOCK
        o_r, l_r = ref["out"][0], ref["lse"][0]
        if not dense:
            kept = admissible_set(res["sel"][b, h], ref["scores"][0, 0], nb, cfg.top_k)
            if nb > cfg.top_k:
                qg = inp.q[b, h * G:(h + 1) * G].double().numpy()
                rp = W.row_problem(inp, b, h)
                c32 = O.centroids(rp["k_pages"], list(range(nb - 1)), "f32")[:, 0]
                cents = (O.round_to_bf16(c32) if dt == "bf16" else c32).astype(np.float64)
                s_ref = O.group_scores(qg, cents)
                bound = SCORE_REL * (np.abs(cents) @ np.abs(qg).sum(axis=0)) + 1e-30
                diff = np.abs(res["scores"][b, h, :nb - 1] - s_ref)
                assert np.all(diff <= bound), f"row {(b, h)}: score error {diff.max()}"
                if dt == "bf16" and O.select_blocks(s_ref, nb, cfg.top_k) != kept:
                    stats["bf16_rank_diff"] += 1
            if kept != [int(x) for x in ref["sel"][0, 0] if x >= 0]:
                # a near tie at the cut: the oracle's attention over the admissible set the
                # GPU kept
                stats["near_tie_rows"] += 1
                rp = W.row_problem(inp, b, h)
                kk, vv = O.row_tokens(rp["k_pages"], rp["v_pages"], rp["block_table"][0], L,
                                      kept, 0)
                o_r, l_r = O.attend(rp["q"][0], kk, vv, cfg.sm_scale)
        o_g = res["out"][b, h * G:(h + 1) * G].astype(np.float64)
        err = np.abs(o_g - o_r)
        assert np.isfinite(o_g).all(), f"row {(b, h)}: non-finite output"
        assert err.max() <= OUT_MAX_ABS[dt], f"row {(b, h)}: max-abs {err.max()}"
        assert err.mean() <= OUT_MEAN_ABS[dt], f"row {(b, h)}: mean-abs {err.mean()}"
        lerr = np.abs(res["lse"][b, h * G:(h + 1) * G] - l_r)
        assert lerr.max() <= LSE_ABS[dt], f"row {(b, h)}: lse error {lerr.max()}"
        stats["rows"] += 1
        stats["max_abs"] = max(stats["max_abs"], float(err.max()))
        stats["max_lse"] = max(stats["max_lse"], float(lerr.max()))
    return stats


def all_rows(cfg):
    return [(b, h) for b in range(cfg.batch) for h in range(cfg.num_kv_heads)]


def check_centroids(inp: W.Inputs, cents: torch.Tensor, pages) -> None:
    """Bit-exact centroid comparison for the listed physical pages (both planes of a bf16
    table: the mean and its residual, each rounded to bf16)."""
    cfg = inp.cfg
    pages = list(pages)
    idx = torch.tensor(pages, dtype=torch.int64, device=cents.device)
    if cfg.dtype == "bf16":
        got = [cents[0][idx].float().cpu().numpy(), cents[1][idx].float().cpu().numpy()]
    else:
        got = [cents[idx].float().cpu().numpy()]
    for i0 in range(0, len(pages), 4096):
        chunk = pages[i0:i0 + 4096]
        kp = inp.k_pages[torch.tensor(chunk)].float().numpy()
        want = (list(O.centroid_pair(kp, list(range(len(chunk))))) if cfg.dtype == "bf16"
                else [O.centroids(kp, list(range(len(chunk))), "f32")])
        for plane, (g_all, ref) in enumerate(zip(got, want)):
            g = g_all[i0:i0 + len(chunk)]
            assert np.array_equal(g.view(np.uint32), ref.view(np.uint32)), \
                f"centroid plane {plane} mismatch at {np.argwhere(g != ref)[:3]}"


def oracle_centroid_table(inp: W.Inputs, chunk: int = 4096) -> np.ndarray:
    """fp32 centroids of every physical page (the oracle's, page by page in chunks)."""
    P = inp.num_pages
    out = np.empty((P, inp.cfg.num_kv_heads, inp.cfg.head_dim), dtype=np.float32)
    for p0 in range(0, P, chunk):
        p1 = min(P, p0 + chunk)
        kp = inp.k_pages[p0:p1].float().numpy()
        out[p0:p1] = O.centroids(kp, list(range(p1 - p0)), "f32")
    return out


def selection_report(inp: W.Inputs, sel: np.ndarray, c32: np.ndarray) -> dict:
    """Every row's kept list against the oracle's fp32-centroid selection: counts of rows
    outside the admissible sets (with the first few), of near ties (admissible, not the
    oracle's own set) and of rows whose kept set differs from the ranking by bf16-rounded
    centroids."""
    cfg = inp.cfg
    G, k = cfg.group, cfg.top_k
    rep = dict(rows=0, outside=0, bad=[], near_tie=0, bf16_rank_diff=0)
    q = inp.q.double().numpy()
    for b in range(cfg.batch):
        L = int(inp.seq_lens[b])
        nb = (L + W.BLOCK - 1) // W.BLOCK
        pages = inp.block_table[b, :max(nb - 1, 0)].numpy().astype(np.int64)
        for h in range(cfg.num_kv_heads):
            rep["rows"] += 1
            g = [int(x) for x in sel[b, h] if x >= 0]
            if nb <= k:
                if g != list(range(nb)):
                    rep["outside"] += 1
                    rep["bad"].append((b, h))
                continue
            qg = q[b, h * G:(h + 1) * G]
            cent = c32[pages, h].astype(np.float64)
            s = O.group_scores(qg, cent)
            try:
                kept = admissible_set(sel[b, h], s, nb, k)
            except AssertionError:
                rep["outside"] += 1
                if len(rep["bad"]) < 5:
                    rep["bad"].append((b, h))
                continue
            if kept != O.select_blocks(s, nb, k):
                rep["near_tie"] += 1
            if cfg.dtype == "bf16":
                s16 = O.group_scores(qg, O.round_to_bf16(c32[pages, h]).astype(np.float64))
                if O.select_blocks(s16, nb, k) != kept:
                    rep["bf16_rank_diff"] += 1
    return rep


def compare_token_rows(inp: W.Inputs, res: dict, budget: int, rows) -> dict:
    """Compare a token-level top-k result with oracle.tokentopk row by row.

    Scores: |s_gpu - s| <= SCORE_REL * sum_{g,i} |q_gi k_ti| (the kernel's group-summed fp32
    query and 128-term fp32 dot product against the fp64 oracle).  Selection: admissible
    (oracle.token_admissible) with tol = twice the row's largest score bound, ascending,
    -1 padded.  Outputs: the oracle's attention over the GPU's kept set, within the bf16
    bars."""
    cfg = inp.cfg
    G = cfg.group
    stats = dict(rows=0, near_tie_rows=0, short_rows=0, max_abs=0.0)
    for b, h in rows:
        rp = W.row_problem(inp, b, h)
        L = int(inp.seq_lens[b])
        qg = rp["q"][0].astype(np.float64)
        kk, vv = O.row_keys_values(rp["k_pages"], rp["v_pages"], rp["block_table"][0], L, 0)
        s = O.token_scores(qg, kk)
        bound = SCORE_REL * (np.abs(kk) @ np.abs(qg).sum(axis=0)) + 1e-30
        sg = res["scores"][b, h, :L].astype(np.float64)
        assert np.all(np.abs(sg - s) <= bound), f"row {(b, h)}: score error {np.abs(sg - s).max()}"
        got = res["sel"][b, h]
        n_keep = min(L, budget)
        kept = [int(t) for t in got[:n_keep]]
        assert all(int(t) == -1 for t in got[n_keep:]), f"row {(b, h)}: padding {got[n_keep:]}"
        assert kept == sorted(kept), f"row {(b, h)}: kept positions not ascending"
        assert O.token_admissible(s, kept, budget, 2.0 * float(bound.max())), \
            f"row {(b, h)}: kept set not admissible"
        if kept != O.select_tokens(s, budget):
            stats["near_tie_rows"] += 1
        stats["short_rows"] += L <= budget
        o_r, l_r = O.attend(qg, kk[kept], vv[kept], cfg.sm_scale)
        o_g = res["out"][b, h * G:(h + 1) * G].astype(np.float64)
        err = np.abs(o_g - o_r)
        assert np.isfinite(o_g).all(), f"row {(b, h)}: non-finite output"
        assert err.max() <= OUT_MAX_ABS["bf16"] and err.mean() <= OUT_MEAN_ABS["bf16"], \
            f"row {(b, h)}: output error {err.max()} / {err.mean()}"
        lerr = np.abs(res["lse"][b, h * G:(h + 1) * G] - l_r)
        assert lerr.max() <= LSE_ABS["bf16"], f"row {(b, h)}: lse error {lerr.max()}"
        stats["rows"] += 1
        stats["max_abs"] = max(stats["max_abs"], float(err.max()))
    return stats
