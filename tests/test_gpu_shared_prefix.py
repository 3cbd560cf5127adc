"""The shared-prefix hint of the Best-of-N decode (kin_decode_args.shared_prefix_blocks):
the leading blocks every sample shares are read with an L2 evict-last policy, so that HBM
serves each shared page once per step for all samples.  It is a cache hint only, so every
result must be bit-identical with and without it: kept lists, scores, outputs, lse and the
appended centroids, for block top-k and for dense decode, and the block top-k result must
still match the oracle.
"""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from _gpu import DeviceState, all_rows, compare_rows  # noqa: E402


def _best_of_n(batch=24, prefix=512, lo=600, hi=3000, seed=21):
    cfg = W.find_config("best-of-n-qwen3-14b")
    return cfg.scaled(batch=batch, prefix=prefix, ctx_lo=lo, ctx_hi=hi, seed=seed, steps=1)


@pytest.mark.parametrize("dense", [False, True])
def test_shared_prefix_hint_changes_no_result(dense):
    cfg = _best_of_n()
    inp = W.generate(cfg)
    shared = cfg.prefix // W.BLOCK
    plain = DeviceState(inp, append=False)
    hinted = DeviceState(inp, append=False)
    a = plain.decode(dense=dense, append_final=True)
    b = hinted.decode(dense=dense, append_final=True, shared_prefix_blocks=shared)
    assert plain.error_bits() == 0 and hinted.error_bits() == 0
    for key in a:
        assert np.array_equal(a[key], b[key], equal_nan=True), key
    assert torch.equal(plain.cents, hinted.cents)
    if not dense:
        stats = compare_rows(inp, b, all_rows(cfg)[::5])
        assert stats["rows"] > 0


def test_shared_prefix_hint_covering_every_block():
    """The hint may name every block of the table (all pages kept in L2)."""
    cfg = _best_of_n(batch=8, prefix=256, lo=100, hi=400)
    inp = W.generate(cfg)
    st = DeviceState(inp)
    a = st.decode()
    b = st.decode(shared_prefix_blocks=inp.max_blocks)
    assert st.error_bits() == 0
    for key in a:
        assert np.array_equal(a[key], b[key], equal_nan=True), key
