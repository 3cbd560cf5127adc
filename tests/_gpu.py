"""Helpers for the GPU parity tests: upload seeded inputs, run the library through its
C ABI binding, and compare with the CPU oracle row by row.

Tolerances:
* bf16 outputs: max-abs 2e-2 and mean-abs 2e-3 per row (the acceptance bar of the
  method's specification); lse within 2e-3 (the kernel rounds each softmax weight to
  bf16 before summing it, a relative error of at most 2^-9 in the sum, i.e. 2e-3 in ln).
* fp32 outputs: max-abs 1e-4, lse 1e-5 (fp32 accumulation and exp2 over <= 2^14 terms).
* Centroids: bit-exact (both sides sum the 16 keys in fp32 in token order and round the
  mean to the stored type the same way).
* Scores: |s_gpu - s_oracle| <= 2e-5 * sum_{g,i} |q_gi c_i| (fp32 dot products of <= 2048
  terms against an fp64 reference).
* Selection: bit-exact, except where the oracle's last kept and first dropped candidate
  scores differ by less than 1e-3 relative; then every block on which the two sides
  disagree must lie within that band, and the row's output is not compared (it is not
  unique).
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
        self.cents = torch.zeros((inp.num_pages, cfg.num_kv_heads, cfg.head_dim),
                                 dtype=W.torch_dtype(cfg.dtype), device=dev)
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

    def decode(self, dense=False, append_final=False):
        cfg = self.inp.cfg
        B, Hq, H = cfg.batch, cfg.num_q_heads, cfg.num_kv_heads
        out = torch.full((B, Hq, cfg.head_dim), float("nan"), dtype=self.q.dtype, device=self.dev)
        lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=self.dev)
        if dense:
            K.dense_decode(self.cache, self.q, self.table, self.lens, cfg.sm_scale, out=out,
                           lse=lse, err_flag=self.err, centroids=self.cents,
                           append_final=append_final)
            torch.cuda.synchronize()
            return dict(out=out.float().cpu().numpy(), lse=lse.cpu().numpy())
        sel = torch.full((B, H, cfg.top_k), -7, dtype=torch.int32, device=self.dev)
        scores = torch.full((B, H, self.inp.max_blocks), float("nan"), dtype=torch.float32,
                            device=self.dev)
        K.blocktopk_decode(self.cache, self.q, self.table, self.lens, self.cents, cfg.top_k,
                           cfg.sm_scale, out=out, lse=lse, sel_blocks=sel, scores=scores,
                           err_flag=self.err, append_final=append_final)
        torch.cuda.synchronize()
        return dict(out=out.float().cpu().numpy(), lse=lse.cpu().numpy(),
                    sel=sel.cpu().numpy(), scores=scores.cpu().numpy())

    def error_bits(self) -> int:
        torch.cuda.synchronize()
        return int(self.err.item())


def oracle_row(inp: W.Inputs, b: int, h: int, dense: bool) -> dict:
    cfg = inp.cfg
    rp = W.row_problem(inp, b, h)
    store = "bf16" if cfg.dtype == "bf16" else "f32"
    if dense:
        return O.dense_decode(rp["q"], rp["k_pages"], rp["v_pages"], rp["block_table"],
                              rp["seq_lens"], cfg.sm_scale)
    return O.blocktopk_decode(rp["q"], rp["k_pages"], rp["v_pages"], rp["block_table"],
                              rp["seq_lens"], cfg.sm_scale, cfg.top_k, store=store)


def selection_ok(sel_g, sel_o, scores_o, nb, k) -> bool:
    """True when the kept sets agree, or differ only inside the near-tie band."""
    g = [int(x) for x in sel_g if x >= 0]
    o = [int(x) for x in sel_o if x >= 0]
    assert len(g) == min(nb, k) and g == sorted(set(g)) and g[-1] == nb - 1, (g, nb, k)
    if g == o:
        return True
    assert nb > k, "with nb <= k the kept set is every block"
    cand = np.asarray(scores_o[: nb - 1], dtype=np.float64)
    order = sorted(range(nb - 1), key=lambda j: (-cand[j], j))
    t_in, t_out = cand[order[k - 2]], cand[order[k - 1]]
    band = TIE_REL * max(abs(t_in), 1e-30)
    assert abs(t_in - t_out) < band, f"selection differs outside a near-tie: {t_in} vs {t_out}"
    for j in set(g) ^ set(o):
        assert abs(cand[j] - t_in) <= band, f"block {j} differs but is not near the cut"
    return False


def compare_rows(inp: W.Inputs, res: dict, rows, dense=False, q_host=None) -> dict:
    """Compare the GPU result of the listed rows with the oracle; returns statistics."""
    cfg = inp.cfg
    G = cfg.group
    dt = cfg.dtype
    stats = dict(rows=0, near_tie_rows=0, max_abs=0.0, max_lse=0.0)
    for b, h in rows:
        ref = oracle_row(inp, b, h, dense)
        L = int(inp.seq_lens[b])
        nb = (L + W.BLOCK - 1) // W.BLOCK
        exact = True
        if not dense:
            exact = selection_ok(res["sel"][b, h], ref["sel"][0, 0], ref["scores"][0, 0], nb,
                                 cfg.top_k)
            if nb > cfg.top_k:
                qg = inp.q[b, h * G:(h + 1) * G].double().numpy()
                rp = W.row_problem(inp, b, h)
                cents = O.centroids(rp["k_pages"], list(range(nb - 1)),
                                    "bf16" if dt == "bf16" else "f32")[:, 0].astype(np.float64)
                bound = SCORE_REL * (np.abs(cents) @ np.abs(qg).sum(axis=0)) + 1e-30
                diff = np.abs(res["scores"][b, h, :nb - 1] - ref["scores"][0, 0, :nb - 1])
                assert np.all(diff <= bound), f"row {(b, h)}: score error {diff.max()}"
        if not exact:
            stats["near_tie_rows"] += 1
            continue
        o_g = res["out"][b, h * G:(h + 1) * G].astype(np.float64)
        o_r = ref["out"][0]
        err = np.abs(o_g - o_r)
        assert np.isfinite(o_g).all(), f"row {(b, h)}: non-finite output"
        assert err.max() <= OUT_MAX_ABS[dt], f"row {(b, h)}: max-abs {err.max()}"
        assert err.mean() <= OUT_MEAN_ABS[dt], f"row {(b, h)}: mean-abs {err.mean()}"
        lerr = np.abs(res["lse"][b, h * G:(h + 1) * G] - ref["lse"][0])
        assert lerr.max() <= LSE_ABS[dt], f"row {(b, h)}: lse error {lerr.max()}"
        stats["rows"] += 1
        stats["max_abs"] = max(stats["max_abs"], float(err.max()))
        stats["max_lse"] = max(stats["max_lse"], float(lerr.max()))
    return stats


def all_rows(cfg):
    return [(b, h) for b in range(cfg.batch) for h in range(cfg.num_kv_heads)]


def check_centroids(inp: W.Inputs, cents: torch.Tensor, pages) -> None:
    """Bit-exact centroid comparison for the listed physical pages."""
    cfg = inp.cfg
    pages = list(pages)
    store = "bf16" if cfg.dtype == "bf16" else "f32"
    got = cents[torch.tensor(pages, dtype=torch.int64, device=cents.device)].float().cpu().numpy()
    for i0 in range(0, len(pages), 4096):
        chunk = pages[i0:i0 + 4096]
        ref = O.centroids(inp.k_pages[torch.tensor(chunk)].float().numpy(),
                          list(range(len(chunk))), store)
        g = got[i0:i0 + len(chunk)]
        assert np.array_equal(g.view(np.uint32), ref.view(np.uint32)), \
            f"centroid mismatch at {np.argwhere(g != ref)[:3]}"
