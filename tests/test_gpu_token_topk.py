"""GPU parity of the token-level (oracle) top-k decode against the CPU oracle
(oracle.tokentopk): every row at small sizes (several score chunks, attention splits and
16-token tiles, ragged tails, rows shorter than the budget, budgets that are not
multiples of 16, groups of 1 to 16, d 64 and 128) and sampled rows of the four
Qwen3-shaped workloads at full size with the equal-KV budget of 16 tokens per kept
block.

Tolerances (the arithmetic fixes them; tests/_gpu.py compare_token_rows):
* Scores: the kernel sums the group's queries in fp32 and then takes a 128-term fp32 dot
  product; |s_gpu - s| <= 2e-5 * sum_{g,i} |q_gi k_ti| per token (the fp64 oracle is
  exact in comparison).
* Selection: judged by oracle.token_admissible with tol = twice the row's largest score
  bound, so kept sets may differ from the oracle's only on tokens whose exact scores lie
  within that of the B-th largest score.
* Outputs: the oracle's attention over the GPU's kept set, within the bf16 bars of the
  block decode tests (max-abs 2e-2, mean-abs 2e-3, lse 2e-3).
"""
import math

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import block_top_sparse_centroid_b300 as K
    from _gpu import DeviceState, compare_token_rows  # noqa: E402


def _cfg(name, d=128, H=2, G=2, lens=(100, 1000), q_std=None, sm_scale=None, seed=11):
    return W.Config(name, len(lens), H * G, H, d, 4, "bf16", "explicit", 0,
                    q_std=q_std if q_std is not None else 1.0 / math.sqrt(d),
                    sm_scale=sm_scale if sm_scale is not None else 1.0 / math.sqrt(d),
                    shuffled=True, seed=seed, lens=tuple(lens))


def _run(inp, budget, events=None):
    st = DeviceState(inp, build=False)
    res = st.token_decode(budget, events=events)
    assert st.error_bits() == 0
    return res


def _check_rows(inp, res, budget, rows) -> dict:
    return compare_token_rows(inp, res, budget, rows)


def _all(cfg):
    return [(b, h) for b in range(cfg.batch) for h in range(cfg.num_kv_heads)]


@pytest.mark.parametrize("d,G,H,lens,budget", [
    (128, 2, 2, (100, 1000, 1, 16, 17, 1031), 64),    # short rows, partial final pages
    (64, 4, 3, (700, 2049, 33), 100),                  # budget not a multiple of 16
    (128, 16, 1, (2000, 513), 300),                    # 16 query heads per KV head
    (128, 1, 4, (4000, 90), 1),                        # one kept token, one query head
    (64, 8, 2, (5000, 4999), 1024),                    # several attention splits per row
    (128, 5, 2, (600, 37), 1024),                      # every row shorter than the budget
    (128, 2, 2, (12000, 900), 2000),                   # keys in shared memory (8K-25.6K)
    (64, 2, 1, (30000, 2000), 800),                    # 32 keys per thread, 1024 threads
    (64, 2, 1, (40000, 3000), 500),                    # longer than the register-resident select
])
def test_token_topk_parity(d, G, H, lens, budget):
    inp = W.generate(_cfg(f"tok-{d}-{G}-{H}", d=d, H=H, G=G, lens=lens))
    res = _run(inp, budget)
    stats = _check_rows(inp, res, budget, _all(inp.cfg))
    assert stats["rows"] == len(lens) * H


def test_token_topk_offset_chunks():
    """448 rows (one attention CTA each) with 2500 kept tokens: every CTA stages its kept
    tokens' rows in two chunks.  24 sampled rows checked."""
    inp = W.generate(_cfg("tok-chunks", d=64, H=8, G=1, lens=(3000,) * 56))
    res = _run(inp, 2500)
    stats = _check_rows(inp, res, 2500, W.sample_rows(inp.cfg, 24, seed=3))
    assert stats["rows"] == 24


def test_token_topk_sharp_softmax():
    """Q ~ N(0, 1) with scale 1: near one-hot softmax weights exercise the running max."""
    inp = W.generate(_cfg("tok-sharp", lens=(3000, 1500), q_std=1.0, sm_scale=1.0))
    res = _run(inp, 256)
    _check_rows(inp, res, 256, _all(inp.cfg))


def test_token_topk_budget_covering_rows_equals_dense():
    """B >= L keeps every token: the output is dense decode's (both over all tokens)."""
    inp = W.generate(_cfg("tok-dense", lens=(300, 77)))
    res = _run(inp, 512)
    dense = DeviceState(inp).decode(dense=True)
    assert np.abs(res["out"] - dense["out"]).max() <= 4e-3
    for b, L in enumerate((300, 77)):
        assert list(res["sel"][b, 0, :L]) == list(range(L))


def test_token_topk_repeat_calls_and_timed_variant():
    """Calls share the workspace (split counters return to zero) and the timed variant does
    the same work."""
    inp = W.generate(_cfg("tok-repeat", G=8, lens=(6000, 3000), d=64))
    first = _run(inp, 1024)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    second = _run(inp, 1024, events=evs)
    assert np.array_equal(first["sel"], second["sel"])
    assert np.array_equal(first["out"], second["out"])
    times = [evs[i].elapsed_time(evs[i + 1]) for i in range(3)]
    assert all(t >= 0.0 for t in times)


@pytest.mark.parametrize("ci", [1, 2, 3, 4])
def test_token_topk_full_size_sampled_rows(ci):
    """The Qwen3-shaped workloads at full size, budget 16 top_k tokens, 12 sampled rows."""
    cfg = W.CONFIGS[ci]
    inp = W.generate(cfg)
    budget = 16 * cfg.top_k
    res = _run(inp, budget)
    rows = W.sample_rows(cfg, 12, seed=5)
    stats = _check_rows(inp, res, budget, rows)
    print(cfg.name, stats)
    assert stats["rows"] == 12
