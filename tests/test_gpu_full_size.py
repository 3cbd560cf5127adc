"""GPU parity at the four benchmark workloads' full sizes, in the launch configuration the
benchmark times: the same seeded inputs and shapes (so the same launch plan), one block
top-k decode call with the fused centroid append of the pages the current token completed.

Rows of full-size workloads are too many for the oracle to check all of them, so:
* every row: the kept list is valid (ascending, distinct, min(nb, k) blocks, the final
  block last) and admissible against the oracle's fp32-centroid selection (bit-exact, or
  differing only inside the 1e-3 near-tie band); every output and lse is finite;
* a seeded sample of rows (plus the first and the last row): selection, scores, outputs
  and lse against the oracle, one row at a time, with the tolerances of the small-size
  tests (near-tie rows against the oracle's attention over the admissible set kept);
* every appended centroid: bit-exact against the oracle's centroid of that page;
* dense decode (the comparison baseline) on a few sampled rows.
"""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from _gpu import (DeviceState, check_centroids, compare_rows,  # noqa: E402
                      oracle_centroid_table, selection_report)

SAMPLED_ROWS = 12


def _kept_lists_valid(inp, sel):
    cfg = inp.cfg
    k = cfg.top_k
    lens = inp.seq_lens.numpy().astype(np.int64)
    nb = (lens + W.BLOCK - 1) // W.BLOCK
    for b in range(cfg.batch):
        want = min(int(nb[b]), k)
        rows = sel[b]                                      # [H, k]
        kept = rows[:, :want]
        assert np.all(rows[:, want:] == -1), f"sequence {b}: padding of the kept list"
        assert np.all(kept[:, -1] == nb[b] - 1), f"sequence {b}: final block not last"
        assert np.all(kept >= 0) and np.all(kept < nb[b]), f"sequence {b}: block id out of range"
        assert np.all(np.diff(kept, axis=1) > 0), f"sequence {b}: kept list not ascending"


# workload name -> seed of its sampled rows
FULL_SIZE = {"qwen3-0.6b": 1, "qwen3-8b": 2, "qwen3-32b-ragged": 3, "best-of-n-qwen3-14b": 4}


@pytest.mark.parametrize("name", list(FULL_SIZE))
def test_full_size_workload(name):
    cfg = W.find_config(name)
    inp = W.generate(cfg)
    # prefill centroids only; the decode call appends the pages the current token completed
    st = DeviceState(inp, append=False)
    res = st.decode(append_final=True)
    assert st.error_bits() == 0

    _kept_lists_valid(inp, res["sel"])
    assert np.isfinite(res["out"]).all()
    assert np.isfinite(res["lse"]).all()

    rep = selection_report(inp, res["sel"], oracle_centroid_table(inp))
    print(f"{name}: {rep['rows']} rows, {rep['outside']} outside the near-tie band, "
          f"{rep['near_tie']} near ties, {rep['bf16_rank_diff']} differ from the bf16-centroid "
          f"ranking")
    assert rep["outside"] == 0, rep

    rows = W.sample_rows(cfg, SAMPLED_ROWS, seed=FULL_SIZE[name])
    rows = sorted(set(rows) | {(0, 0), (cfg.batch - 1, cfg.num_kv_heads - 1)})
    stats = compare_rows(inp, res, rows)
    assert stats["rows"] == len(rows)

    if st.just_pages:
        check_centroids(inp, st.cents, st.just_pages)

    dense = st.decode(dense=True)
    assert st.error_bits() == 0
    compare_rows(inp, dense, rows[:3], dense=True)
