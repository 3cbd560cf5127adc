"""GPU parity of the selection on the paths the benchmark workloads do not reach.

* Long rows: more candidates than the selecting warp (2048) or CTA (4096 with 8 consumer
  warps, 2048 with 4) holds in registers, up to the largest row the library accepts
  (16383 candidates), with one warp per row (more than two rows per CTA) and with
  cooperative selection (at most two).  Checked against the oracle's fp32-centroid
  selection and attention.
* Rows where only the second centroid code can rank the candidates: every block's mean
  rounds to the same bf16 value, and the fp32 means differ by more than the near-tie band.
  A selection from the first code alone would keep the lowest indices; the library must
  keep the oracle's blocks exactly, on every path (ambiguous candidates re-scored from the
  selection's shared-memory list of 256, and more of them than the list holds).
"""
import math

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from _gpu import (DeviceState, all_rows, compare_rows, oracle_centroid_table,  # noqa: E402
                      selection_report)


def _cfg(name, lens, H, G, d=128, k=16, seed=1, q_std=None):
    return W.Config(name, len(lens), H * G, H, d, k, "bf16", "explicit", 0,
                    q_std=q_std if q_std is not None else 1.0 / math.sqrt(d),
                    sm_scale=1.0 / math.sqrt(d), shuffled=True, seed=seed, lens=tuple(lens))


def _check_all(inp, res, sample=None):
    rep = selection_report(inp, res["sel"], oracle_centroid_table(inp))
    assert rep["outside"] == 0, rep
    rows = all_rows(inp.cfg) if sample is None else W.sample_rows(inp.cfg, sample, seed=3)
    return rep, compare_rows(inp, res, rows)


@pytest.mark.parametrize("case", ["warp_rows", "cta8_rows", "cta4_rows", "max_blocks"])
def test_long_rows(case):
    if case == "warp_rows":
        # 304 rows (> 2 x 148 CTAs): one warp per row, 2062..2499 candidates (> 2048 in
        # registers)
        lens = tuple(33000 + 187 * i for i in range(38))
        cfg = _cfg("long-warp", lens, H=8, G=1, d=64, k=24, seed=31)
        sample = 10
    elif case == "cta8_rows":
        # 2 rows, 8 consumer warps: 4374 and 6249 candidates (> 4096 in registers)
        cfg = _cfg("long-cta8", (70000, 100000), H=1, G=4, k=64, seed=32)
        sample = None
    elif case == "cta4_rows":
        # 2 rows, 4 consumer warps (groups of 16): 2499 and 4374 candidates (> 2048)
        cfg = _cfg("long-cta4", (40000, 70000), H=1, G=16, k=32, seed=33)
        sample = None
    else:
        # the largest accepted row: max_blocks 16384, 16383 candidates
        cfg = _cfg("max-blocks", (262144, 262143), H=1, G=2, k=128, seed=34)
        sample = None
    inp = W.generate(cfg)
    st = DeviceState(inp)
    res = st.decode()
    assert st.error_bits() == 0
    _check_all(inp, res, sample)


def _residual_decides(inp, high_frac_rows, k, seed):
    """Make every candidate block's mean key round to 1.0 (bf16) in dimension 0, with the
    fp32 means at 1 + 2^-10 ("low") or 1 + 3 * 2^-10 ("high"), and queries one-hot on
    dimension 0: the fp32 ranking is the "high" blocks first (then the lowest-index "low"
    ones), which the first code alone cannot see.  The gap, 2^-9 relative, is above the
    near-tie band (1e-3), so the kept set must match the oracle's exactly."""
    g = torch.Generator().manual_seed(seed)
    cfg = inp.cfg
    inp.q.zero_()
    inp.q[:, :, 0] = 1.0
    for b in range(cfg.batch):
        L = int(inp.seq_lens[b])
        nb = (L + 15) // 16
        pages = inp.block_table[b, :nb - 1].long()
        n = nb - 1
        high = torch.zeros(n, dtype=torch.bool)
        n_high = max(0, min(n, k - 1 - 3))      # three more kept from the "low" level, by index
        high[torch.randperm(n, generator=g)[:n_high]] = True
        for h in range(cfg.num_kv_heads):
            kp = inp.k_pages[pages, h]                               # [n, 16, d] (a copy)
            kp[:, :, 0] = 1.0
            # one token of 1 + 2^-6 (low) or 1 + 3 * 2^-6 (high): exact in bf16
            kp[:, 0, 0] = torch.where(high, 1.0 + 3 * 2.0 ** -6, 1.0 + 2.0 ** -6).to(kp.dtype)
            inp.k_pages[pages, h] = kp


@pytest.mark.parametrize("case", ["warp_list", "warp_over_cap", "cta_list", "cta_over_cap"])
def test_second_code_decides_selection(case):
    if case == "warp_list":          # 304 rows, one warp each, 100 ambiguous candidates
        cfg = _cfg("res-warp", (16 * 101,) * 38, H=8, G=2, d=64, k=40, seed=41)
    elif case == "warp_over_cap":    # 304 rows, 600 ambiguous candidates (> 256 listed)
        cfg = _cfg("res-warp-big", (16 * 601,) * 38, H=8, G=1, d=64, k=40, seed=42)
    elif case == "cta_list":         # 4 rows, cooperative, 150-200 ambiguous (<= 256 listed)
        cfg = _cfg("res-cta", (16 * 201, 16 * 150 + 3), H=2, G=4, k=64, seed=43)
    else:                            # 2 rows, cooperative, 2000 ambiguous (> 256 listed)
        cfg = _cfg("res-cta-big", (16 * 2001, 16 * 1500 + 9), H=1, G=8, k=100, seed=44)
    inp = W.generate(cfg)
    _residual_decides(inp, 0.5, cfg.top_k, seed=cfg.seed)
    st = DeviceState(inp)
    res = st.decode()
    assert st.error_bits() == 0
    rep = selection_report(inp, res["sel"], oracle_centroid_table(inp))
    assert rep["outside"] == 0, rep
    assert rep["near_tie"] == 0, rep             # no near ties: the kept sets are the oracle's
    assert rep["bf16_rank_diff"] == rep["rows"]  # the first code alone would pick otherwise
    compare_rows(inp, res, W.sample_rows(cfg, 6, seed=5))
