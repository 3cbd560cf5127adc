"""GPU parity of the best-of-N decode loop: 64 consecutive decode steps over one paged
cache whose samples share the prompt's pages.  Before every step but the first, each
sample's new token is written into its page (torch indexing: the caller's part) and
seq_lens advance; the step is one block top-k decode that also appends the centroid of
every page the token completed, and later steps score those pages.

Checked at every step: each appended centroid, bit for bit (both codes), and that every
kept list is valid.  At steps around page boundaries: sampled rows against the oracle on
the host copy of the same state (selection, scores, outputs, lse), and dense decode on a
few rows.  At the last step: every row's kept list against the oracle's fp32-centroid
selection, and every complete page's centroid.
"""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from _gpu import (DeviceState, check_centroids, compare_rows,  # noqa: E402
                      oracle_centroid_table, selection_report)

CHECK_STEPS = {0, 1, 2, 15, 16, 17, 31, 47, 62, 63}


def _just_completed(inp):
    """Physical pages whose 16th token is each sequence's current one."""
    last = inp.last_pages().tolist()
    return sorted({p for b, p in enumerate(last) if int(inp.seq_lens[b]) % W.BLOCK == 0})


def _kept_valid(inp, sel):
    k = inp.cfg.top_k
    for b in range(inp.cfg.batch):
        nb = (int(inp.seq_lens[b]) + W.BLOCK - 1) // W.BLOCK
        want = min(nb, k)
        kept = sel[b][:, :want]
        assert np.all(sel[b][:, want:] == -1)
        assert np.all(kept[:, -1] == nb - 1)
        assert np.all(np.diff(kept, axis=1) > 0) and np.all(kept >= 0)


def _run_loop(cfg, sample_rows, full_report):
    inp = W.generate(cfg)
    st = DeviceState(inp, append=False)     # prefill: the pages complete before step 0
    dev = st.dev
    appended = 0
    for t in range(cfg.steps):
        if t > 0:
            tok = W.step_tokens(inp, t)
            W.write_step_tokens(inp, tok)                     # host copy of the state
            pages, slots = tok.pages.to(dev), tok.slots.to(dev)
            st.cache.k_pages[pages, :, slots, :] = tok.k_new.to(dev)
            st.cache.v_pages[pages, :, slots, :] = tok.v_new.to(dev)
            st.lens += 1
            st.q = tok.q.to(dev)
        res = st.decode(append_final=True)
        assert st.error_bits() == 0, f"step {t}"
        _kept_valid(inp, res["sel"])
        just = _just_completed(inp)
        if just:
            check_centroids(inp, st.cents, just)
            appended += len(just)
        if t in CHECK_STEPS:
            rows = W.sample_rows(cfg, sample_rows, seed=100 + t)
            stats = compare_rows(inp, res, rows)
            assert stats["rows"] == len(rows)
        if t == cfg.steps - 1:
            dense = st.decode(dense=True)
            compare_rows(inp, dense, W.sample_rows(cfg, 3, seed=7), dense=True)
            if full_report:
                rep = selection_report(inp, res["sel"], oracle_centroid_table(inp))
                print(f"{cfg.name} step {t}: {rep}")
                assert rep["outside"] == 0, rep
    # every complete page's centroid, built before the loop or appended during it
    check_centroids(inp, st.cents, inp.complete_pages().tolist())
    # positions L0 - 1 .. L0 + 62 of every sample: exactly four complete a page
    assert appended == cfg.batch * (cfg.steps // W.BLOCK)
    return inp


def test_best_of_n_loop_reduced():
    cfg = W.find_config("best-of-n-qwen3-14b").scaled(batch=24, ctx_lo=2048, ctx_hi=4096)
    _run_loop(cfg, sample_rows=10, full_report=True)


def test_best_of_n_loop_full_size():
    cfg = W.find_config("best-of-n-qwen3-14b")
    _run_loop(cfg, sample_rows=6, full_report=True)
