"""GPU parity of the CUDA path against the CPU oracle at sizes the oracle finishes in
seconds: every row checked, several tiles per kernel, ragged tails and edge cases."""
import math

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from _gpu import (DeviceState, all_rows, check_centroids, compare_rows)  # noqa: E402


def _cfg(name, dtype="bf16", d=128, H=2, G=2, k=4, lens=(100, 1000), q_std=None,
         sm_scale=None, seed=7, shuffled=True):
    return W.Config(name, len(lens), H * G, H, d, k, dtype, "explicit", 0,
                    q_std=q_std if q_std is not None else 1.0 / math.sqrt(d),
                    sm_scale=sm_scale if sm_scale is not None else 1.0 / math.sqrt(d),
                    shuffled=shuffled, seed=seed, lens=tuple(lens))


def _run(cfg, dense=False):
    inp = W.generate(cfg)
    st = DeviceState(inp)
    res = st.decode(dense=dense)
    stats = compare_rows(inp, res, all_rows(cfg), dense=dense)
    assert st.error_bits() == 0
    return inp, st, res, stats


def test_tiny_config_fp32():
    cfg = W.find_config("tiny")
    inp, st, res, stats = _run(cfg)
    assert stats["rows"] == 1
    check_centroids(inp, st.cents, inp.complete_pages().tolist())
    _run(cfg, dense=True)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 5, 8, 16])
def test_group_and_head_dim(d, G):
    cfg = _cfg(f"g{G}d{d}", d=d, H=2, G=G, k=6, lens=(17, 260, 1023), seed=G * 100 + d)
    _run(cfg)
    _run(cfg, dense=True)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("G", [1, 5])
@pytest.mark.parametrize("copies", [1, 2])
def test_eight_head_ranges(d, G, copies):
    # 8 KV heads: the score stages of a whole 8-head range (four lanes per centroid); 19
    # sequences (152 rows, at most two per CTA): cooperative selection of each row; 38
    # sequences (304 rows, more than two per CTA): one warp selects each row of a range
    lens = (130, 1500, 4097, 2048, 17, 700, 16 * 33, 999, 3000, 64,
            1201, 250, 16 * 90 + 1, 3333, 160, 2222, 801, 47, 1024) * copies
    cfg = _cfg(f"h8g{G}d{d}x{copies}", d=d, H=8, G=G, k=8, lens=lens, seed=G * 10 + d)
    _run(cfg)


@pytest.mark.parametrize("H,copies", [(4, 1), (16, 1), (16, 2)])
def test_other_head_range_widths(H, copies):
    # 4 heads (40 rows): the queries of the range in registers, cooperative selection;
    # 16 heads: queries read from global memory into one shared copy, two pages per score
    # stage; 160 rows: cooperative selection; 320 rows (more than two per CTA): two rows
    # per selecting warp
    lens = (130, 1500, 4097, 700, 2048, 33, 1111, 16 * 50, 2500, 401) * copies
    cfg = _cfg(f"h{H}x{copies}", H=H, G=2, k=8, lens=lens, seed=H)
    _run(cfg)
    _run(cfg, dense=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("q_std", [None, 1.0, 4.0])
def test_softmax_sharpness(dtype, q_std):
    # q_std 1 and 4 make the softmax peaked, so the output tolerance is a real test
    cfg = _cfg("sharp", dtype=dtype, H=3, G=3, k=8, lens=(300, 777, 2048, 5000), q_std=q_std,
               seed=11)
    _run(cfg)
    _run(cfg, dense=True)


def test_edge_lengths():
    # L < 16, L = 16, L = 17, multiples of 16, nb == k, nb == k + 1, long rows
    lens = (1, 2, 15, 16, 17, 31, 32, 33, 16 * 8, 16 * 8 + 1, 16 * 9, 4096, 4097)
    cfg = _cfg("edges", H=2, G=4, k=8, lens=lens, seed=3)
    _run(cfg)
    _run(cfg, dense=True)


@pytest.mark.parametrize("k", [1, 2, 3, 64, 400])
def test_topk_values(k):
    cfg = _cfg(f"k{k}", H=2, G=2, k=k, lens=(50, 1600, 4000, 6400), seed=k)
    inp, st, res, stats = _run(cfg)
    for b in range(cfg.batch):
        nb = (int(inp.seq_lens[b]) + 15) // 16
        for h in range(cfg.num_kv_heads):
            kept = [x for x in res["sel"][b, h] if x >= 0]
            assert len(kept) == min(nb, k) and kept[-1] == nb - 1
            assert all(x == -1 for x in res["sel"][b, h][len(kept):])


def test_topk_at_least_blocks_equals_dense():
    cfg = _cfg("kbig", H=2, G=4, k=64, lens=(100, 1024, 999), seed=5)
    inp = W.generate(cfg)
    st = DeviceState(inp)
    sp = st.decode()
    de = st.decode(dense=True)
    # with nb <= k both calls read exactly the same tokens in the same order
    assert np.array_equal(sp["out"], de["out"])
    assert np.array_equal(sp["lse"], de["lse"])


def test_unshuffled_and_shared_pages():
    # best-of-N layout: every sample shares the prompt's pages
    cfg = W.find_config("best-of-n-qwen3-14b").scaled(batch=6, ctx_lo=300, ctx_hi=900, prefix=256, steps=1)
    inp, st, res, stats = _run(cfg)
    assert stats["rows"] == cfg.batch * cfg.num_kv_heads


def test_duplicate_blocks_tie_to_lower_index():
    cfg = _cfg("dup", H=1, G=2, k=2, lens=(16 * 6 + 3,), seed=9)
    inp = W.generate(cfg)
    tab = inp.block_table[0]
    # copy block 1's keys into block 4: equal centroids, equal scores
    inp.k_pages[int(tab[4])] = inp.k_pages[int(tab[1])]
    inp.q[0] = inp.q[0] * 0  # all scores equal (zero): ties everywhere
    st = DeviceState(inp)
    res = st.decode()
    assert list(res["sel"][0, 0]) == [0, 6]
    inp.q[0, :, :] = 0
    inp.q[0, 0, 0] = 1.0
    # make block 1 (and its copy, 4) the best: give them a large first key coordinate
    for j in (1, 4):
        inp.k_pages[int(tab[j]), 0, :, 0] = 50.0
    st = DeviceState(inp)
    res = st.decode()
    assert list(res["sel"][0, 0]) == [1, 6]
    compare_rows(inp, res, [(0, 0)])


def test_page_permutation_invariance():
    cfg = _cfg("perm", H=2, G=4, k=5, lens=(900, 333), seed=21, shuffled=True)
    a = W.generate(cfg)
    b = W.generate(cfg)
    perm = torch.randperm(a.num_pages, generator=torch.Generator().manual_seed(5))
    inv = torch.argsort(perm)
    b.k_pages, b.v_pages, b.k_offset = a.k_pages[perm], a.v_pages[perm], a.k_offset[perm]
    b.block_table = torch.where(a.block_table >= 0, inv[a.block_table.clamp(min=0).long()].int(),
                                a.block_table)
    ra, rb = DeviceState(a).decode(), DeviceState(b).decode()
    for key in ("out", "lse", "sel"):
        assert np.array_equal(ra[key], rb[key]), key


def test_repeat_calls_identical_and_dirty_workspace():
    cfg = _cfg("rep", H=8, G=2, k=8, lens=(4000,) * 8, seed=2)
    inp = W.generate(cfg)
    st = DeviceState(inp)
    r1 = st.decode()
    r2 = st.decode()
    d1 = st.decode(dense=True)
    d2 = st.decode(dense=True)
    for key in ("out", "lse", "sel", "scores"):
        assert np.array_equal(r1[key], r2[key], equal_nan=True), key
    assert np.array_equal(d1["out"], d2["out"])
    # every call leaves the workspace's counter area zero, whatever the shapes, so calls
    # of other shapes (whose data regions cover other bytes) may share it in between
    import block_top_sparse_centroid_b300.api as A
    buf = A._default_ws[(st.dev.type, st.dev.index)].buf
    assert int(buf[:65536].count_nonzero()) == 0
    other = DeviceState(W.generate(_cfg("rep2", H=2, G=4, k=4, lens=(900, 70, 3000), seed=3)))
    other.decode()
    other.decode(dense=True)
    assert A._default_ws[(st.dev.type, st.dev.index)].buf is buf   # no regrowth: same bytes reused
    assert int(buf[:65536].count_nonzero()) == 0
    r3 = st.decode()
    for key in ("out", "lse", "sel", "scores"):
        assert np.array_equal(r1[key], r3[key], equal_nan=True), key


def test_centroid_build_all_pages_and_append():
    cfg = _cfg("cent", H=3, G=2, k=4, lens=(160, 48, 1600), seed=4)
    inp = W.generate(cfg, poison=False)
    st = DeviceState(inp, build=False)
    import block_top_sparse_centroid_b300 as K
    K.centroids_build(st.cache, st.cents, err_flag=st.err)       # every page
    torch.cuda.synchronize()
    check_centroids(inp, st.cents, range(inp.num_pages))
    # append: recompute a few pages after changing their keys
    pages = [int(inp.block_table[2, j]) for j in (0, 5, 99)]
    for p in pages:
        inp.k_pages[p] = -inp.k_pages[p]
        st.cache.k_pages[p] = inp.k_pages[p].to(st.dev)
    K.centroids_append(st.cache, torch.tensor(pages, dtype=torch.int32, device=st.dev), st.cents)
    torch.cuda.synchronize()
    check_centroids(inp, st.cents, range(inp.num_pages))
    assert st.error_bits() == 0


def test_device_error_flags_without_fault():
    cfg = _cfg("bad", H=2, G=2, k=3, lens=(200, 300, 64), seed=8)
    inp = W.generate(cfg)
    st = DeviceState(inp)
    # a block-table entry outside the page pool (kept block: the final one) and a
    # sequence length of 0: the kernels flag both and skip the data
    st.table[0, (200 + 15) // 16 - 1] = inp.num_pages + 12345
    st.lens[2] = 0
    res = st.decode()
    bits = st.error_bits()
    assert bits & 1 and bits & 2
    assert np.all(res["out"][2] == 0) and np.all(np.isneginf(res["lse"][2]))
    assert np.all(np.isfinite(res["out"][:2]))
    # the untouched sequence is still right
    compare_rows(inp, res, [(1, 0), (1, 1)])
    # centroid build with an out-of-range page id
    import block_top_sparse_centroid_b300 as K
    st.err.zero_()
    K.centroids_build(st.cache, st.cents,
                      page_ids=torch.tensor([0, -5, inp.num_pages], dtype=torch.int32,
                                            device=st.dev), err_flag=st.err)
    assert st.error_bits() == 1


def test_dense_multi_split_long_rows():
    # long rows force several attention splits per row and the last-arriver merge
    cfg = _cfg("long", H=1, G=8, k=16, lens=(16384, 9001, 16 * 700 + 5), seed=13)
    _run(cfg, dense=True)
    _run(cfg)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("f32", 64)])
@pytest.mark.parametrize("dense", [False, True])
def test_decode_appends_completed_final_blocks(dtype, d, dense):
    # sequences whose current token completed their final page (L % 16 == 0) and others
    lens = (32, 48, 1600, 1601, 16 * 77, 16 * 3 + 5)
    cfg = _cfg("app", dtype=dtype, d=d, H=2, G=4, k=8, lens=lens, seed=17 + d)
    inp = W.generate(cfg)
    st = DeviceState(inp, append=False)         # final pages' centroids not built yet
    assert st.just_pages
    idx = torch.tensor(st.just_pages, device=st.dev).long()
    zero = st.cents[:, idx] if dtype == "bf16" else st.cents[idx]   # bf16: both planes
    assert int(zero.float().abs().sum()) == 0
    res = st.decode(dense=dense, append_final=True)
    torch.cuda.synchronize()
    check_centroids(inp, st.cents, st.just_pages)
    check_centroids(inp, st.cents, inp.complete_pages().tolist())
    compare_rows(inp, res, all_rows(cfg), dense=dense)
    assert st.error_bits() == 0


def test_many_equal_scores_take_lowest_indices():
    # every candidate block has the same keys, so every score ties: more tied candidates
    # than a warp holds at the cut (the selection's general path), lowest indices kept
    cfg = _cfg("ties", H=2, G=2, k=8, lens=(16 * 100 + 3, 16 * 40), seed=19)
    inp = W.generate(cfg)
    for b in range(cfg.batch):
        nb = (int(inp.seq_lens[b]) + 15) // 16
        tab = inp.block_table[b]
        for j in range(1, nb - 1):
            inp.k_pages[int(tab[j])] = inp.k_pages[int(tab[0])]
    st = DeviceState(inp)
    res = st.decode()
    for b in range(cfg.batch):
        nb = (int(inp.seq_lens[b]) + 15) // 16
        for h in range(cfg.num_kv_heads):
            assert list(res["sel"][b, h]) == list(range(cfg.top_k - 1)) + [nb - 1]
    compare_rows(inp, res, all_rows(cfg))
