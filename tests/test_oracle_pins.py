"""Pins of the CPU oracle against things other than itself (CPU only).

Each pin checks one oracle function against a library routine, a closed form, a brute
force enumeration, an invariant, or a number printed on the pages (tests/golden/).  The
mutation tests at the end plant plausible mistakes in the oracle and check that at
least one pin fails for each, so a mistake of that kind cannot hide.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle.blocktopk as OB

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
U32 = 2.0 ** -24


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16_exact(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy()


# ----------------------------------------------------------------------------- bf16 code
def pin_bf16_rounding():
    """round_to_bf16 equals torch's float32 -> bfloat16 conversion bit for bit."""
    r = _rng(1)
    vals = [r.standard_normal(20000).astype(np.float32),
            (r.standard_normal(20000) * 10.0 ** r.integers(-30, 30, 20000)).astype(np.float32)]
    hi = r.integers(0, 1 << 16, 4000, dtype=np.uint64)
    halfway = ((hi << np.uint64(16)) | np.uint64(0x8000)).astype(np.uint32).view(np.float32)
    vals.append(halfway[np.isfinite(halfway)])
    vals.append(np.array([0.0, -0.0, 1e-40, -1e-40, 3.4e38, -3.4e38, np.inf, -np.inf],
                         dtype=np.float32))
    x = np.concatenate(vals).astype(np.float32)
    got = OB.round_to_bf16(x)
    ref = torch.tensor(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert np.isnan(OB.round_to_bf16(np.array([np.nan], np.float32)))[0]


# ----------------------------------------------------------------------------- centroid
def pin_centroid_closed_forms():
    r = _rng(2)
    d = 32
    # 16 copies of one bf16-representable row: the mean is the row itself.
    row = _bf16_exact(r.standard_normal(d))
    blk = np.repeat(row[None, :], 16, axis=0)
    assert np.array_equal(OB.block_centroid(blk, "f32"), row)
    assert np.array_equal(OB.block_centroid(blk, "bf16"), row)
    # integer keys: every partial sum is exact, so the mean is the exact rational mean.
    ik = r.integers(-100, 101, (16, d)).astype(np.float32)
    exact = [Fraction(int(ik[:, i].sum()), 16) for i in range(d)]
    c = OB.block_centroid(ik, "f32")
    assert all(Fraction(float(c[i])) == exact[i] for i in range(d))
    # general keys: within the first-order bound of 15 float32 roundings of the sum.
    for trial in range(20):
        kk = (r.standard_normal((16, d)) * 10.0 ** r.uniform(-3, 3)).astype(np.float32)
        c32 = OB.block_centroid(kk, "f32")
        for i in range(d):
            mean = math.fsum(float(v) for v in kk[:, i]) / 16.0
            bound = 15 * U32 * sum(abs(float(v)) for v in kk[:, i]) / 16.0 * 1.01
            assert abs(float(c32[i]) - mean) <= bound + 1e-45
        cb = OB.block_centroid(kk, "bf16")
        assert np.array_equal(cb, _bf16_exact(c32))
    # the batched form agrees with the single-block form for every page and head
    pages = r.standard_normal((5, 3, 16, d)).astype(np.float32)
    allc = OB.centroids(pages, [4, 0, 2], "bf16")
    for n, p in enumerate([4, 0, 2]):
        for h in range(3):
            assert np.array_equal(allc[n, h], OB.block_centroid(pages[p, h], "bf16"))


def pin_centroid_pair():
    """The bf16 (hi, lo) code of a centroid: hi is the fp32 mean rounded to bf16, lo the
    exact residual rounded to bf16, and hi + lo is the fp32 mean to 2^-16 of its size."""
    # closed form: fifteen keys 1.0 and one 1 + 2^-6 (both exact in bf16) have the mean
    # 1 + 2^-10, which bf16 (7 fraction bits) rounds to 1: hi = 1 and lo = 2^-10 exactly
    keys = np.ones((16, 4), dtype=np.float32)
    keys[7, :] = 1.0 + 2.0 ** -6
    hi, lo = OB.centroid_pair(keys[None, None], [0])
    assert np.all(hi == 1.0) and np.all(lo == 2.0 ** -10)
    # a mean that bf16 holds exactly has no residual
    keys = np.full((16, 4), 0.75, dtype=np.float32)
    hi, lo = OB.centroid_pair(keys[None, None], [0])
    assert np.all(hi == 0.75) and np.all(lo == 0.0)
    r = _rng(12)
    pages = (r.standard_normal((6, 2, 16, 48)) * 10.0 ** r.uniform(-3, 3, (6, 1, 1, 1))).astype(np.float32)
    pages = _bf16_exact(pages)
    hi, lo = OB.centroid_pair(pages, [5, 0, 3])
    for n, p in enumerate([5, 0, 3]):
        for h in range(2):
            c32 = OB.block_centroid(pages[p, h], "f32")
            assert np.array_equal(hi[n, h], _bf16_exact(c32))
            diff64 = c32.astype(np.float64) - hi[n, h].astype(np.float64)
            assert np.array_equal(diff64, (c32 - hi[n, h]).astype(np.float64))  # exact in fp32
            assert np.array_equal(lo[n, h], _bf16_exact(diff64.astype(np.float32)))
            err = np.abs(c32.astype(np.float64) - hi[n, h] - lo[n, h].astype(np.float64))
            assert np.all(err <= 2.0 ** -16 * np.abs(c32.astype(np.float64)))
            assert np.all(np.abs(diff64) <= 2.0 ** -8 * np.abs(hi[n, h].astype(np.float64)))


def _admissible_by_rule(scores, nb, k, rel):
    """Every kept set of size k that holds the final block and differs from the oracle's
    own only on blocks whose score is within rel of the oracle's last kept score."""
    base = OB.select_blocks(scores, nb, k)
    if nb <= k:
        return [base]
    kept_scores = sorted((float(scores[j]) for j in base[:-1]), reverse=True)
    t = kept_scores[-1] if kept_scores else None
    out = []
    for comb in itertools.combinations(range(nb - 1), k - 1):
        cand = sorted(list(comb) + [nb - 1])
        if all(abs(float(scores[j]) - t) <= rel * abs(t) for j in set(cand) ^ set(base)):
            out.append(cand)
    return out


def pin_valid_selections():
    """The admissible kept sets equal a filter of every subset by the acceptance rule."""
    assert OB.valid_selections([5.0, 5.0, 5.0], 4, 2) == [[0, 3], [1, 3], [2, 3]]
    assert OB.valid_selections([1.0, 9.0, 4.0], 4, 3) == [[1, 2, 3]]      # no near tie
    assert OB.valid_selections([1.0, 9.0], 3, 5) == [[0, 1, 2]]           # nb <= k
    r = _rng(13)
    for trial in range(300):
        nb = int(r.integers(2, 10))
        k = int(r.integers(1, 6))
        base = r.integers(1, 6, nb - 1).astype(np.float64) * 1000.0
        jitter = r.choice([0.0, 1e-4, 5e-4, 2e-3, 1e-2], nb - 1)
        scores = list(base * (1.0 + jitter * r.choice([-1.0, 1.0], nb - 1)))
        got = OB.valid_selections(scores, nb, k)
        want = _admissible_by_rule(scores, nb, k, 1e-3)
        assert sorted(got) == sorted(want), (scores, nb, k)
        assert OB.select_blocks(scores, nb, k) in got


# ----------------------------------------------------------------------------- scores
def pin_group_scores():
    r = _rng(3)
    for G in (1, 2, 5, 8):
        q = r.standard_normal((G, 24))
        c = r.standard_normal((40, 24))
        s = OB.group_scores(q, c)
        ref = np.matmul(c, q.sum(axis=0))        # sum over the group first, then one matmul
        assert np.allclose(s, ref, rtol=1e-12, atol=1e-12)
        # one-hot queries pick single centroid coordinates
        idx = r.integers(0, 24, G)
        oh = np.zeros((G, 24))
        oh[np.arange(G), idx] = 1.0
        assert np.array_equal(OB.group_scores(oh, c), c[:, idx].sum(axis=1))


# ----------------------------------------------------------------------------- selection
def _brute_force_select(scores, nb, k):
    if nb <= k:
        return list(range(nb))
    best, best_set = None, None
    for comb in itertools.combinations(range(nb - 1), k - 1):  # lexicographic order
        tot = sum(scores[j] for j in comb)
        if best is None or tot > best:
            best, best_set = tot, comb
    return sorted(list(best_set) + [nb - 1])


def pin_selection_brute_force():
    r = _rng(4)
    for trial in range(400):
        nb = int(r.integers(1, 11))
        k = int(r.integers(1, 7))
        scores = [int(v) for v in r.integers(-2, 3, max(nb - 1, 0))]  # many exact ties
        got = OB.select_blocks(scores, nb, k)
        assert got == _brute_force_select(scores, nb, k), (scores, nb, k, got)
        assert len(got) == min(nb, k) and got == sorted(set(got)) and got[-1] == nb - 1
    assert OB.select_blocks([5.0, 5.0, 5.0], 4, 2) == [0, 3]          # tie -> lower index
    assert OB.select_blocks([0.0, -0.0, 0.0], 4, 3) == [0, 1, 3]      # -0.0 ties +0.0
    assert OB.select_blocks([1.0, 9.0], 3, 1) == [2]                  # k = 1: final block only


# ----------------------------------------------------------------------------- attention
def pin_attention_vs_sdpa():
    r = _rng(5)
    for G, T, d in ((1, 1, 8), (2, 37, 16), (5, 130, 64), (8, 16, 128)):
        q = r.standard_normal((G, d))
        kk = r.standard_normal((T, d)) * 2.0
        vv = r.standard_normal((T, d))
        sc = 1.0 / math.sqrt(d)
        o, lse = OB.attend(q, kk, vv, sc)
        tq, tk, tv = (torch.tensor(a, dtype=torch.float64) for a in (q, kk, vv))
        ref = torch.nn.functional.scaled_dot_product_attention(
            tq[None, :, None, :], tk[None, None].expand(1, G, T, d),
            tv[None, None].expand(1, G, T, d), scale=sc)[0, :, 0, :].numpy()
        ref_lse = torch.logsumexp(sc * (tq @ tk.T), dim=1).numpy()
        assert np.allclose(o, ref, rtol=1e-12, atol=1e-12)
        assert np.allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)
        # every output is a convex combination of the value rows
        assert np.all(o <= vv.max(axis=0) + 1e-12) and np.all(o >= vv.min(axis=0) - 1e-12)
    # closed form: logits 0 and ln 3 give weights 1/4 and 3/4
    o, lse = OB.attend(np.array([[math.log(3.0)]]), np.array([[0.0], [1.0]]),
                       np.array([[4.0], [8.0]]), 1.0)
    assert abs(o[0, 0] - 7.0) < 1e-14 and abs(lse[0] - math.log(4.0)) < 1e-14


# ----------------------------------------------------------------------------- full step
def _tiny_problem(seed, B=2, H=2, G=3, d=16, k=3, lens=(57, 100), shuffle=True):
    r = _rng(seed)
    nbs = [(L + 15) // 16 for L in lens]
    P = sum(nbs)
    ids = r.permutation(P) if shuffle else np.arange(P)
    table = np.full((B, max(nbs)), -1, dtype=np.int64)
    pos = 0
    for b, n in enumerate(nbs):
        table[b, :n] = ids[pos:pos + n]
        pos += n
    k_pages = (r.standard_normal((P, H, 16, d)) + r.standard_normal((P, H, 1, d))).astype(np.float32)
    v_pages = r.standard_normal((P, H, 16, d)).astype(np.float32)
    for b, L in enumerate(lens):                      # stale slots past the length
        p = table[b, nbs[b] - 1]
        t0 = L - 16 * (nbs[b] - 1)
        k_pages[p, :, t0:] = 1e3
        v_pages[p, :, t0:] = -1e3
    q = r.standard_normal((B, H * G, d)).astype(np.float32)
    return dict(q=q, k_pages=k_pages, v_pages=v_pages, block_table=table,
                seq_lens=np.array(lens, dtype=np.int64)), k


def pin_decode_against_masked_sdpa():
    """Brute-force selection + masked SDPA over the whole sequence equals the oracle."""
    for seed in range(6):
        prob, k = _tiny_problem(10 + seed)
        q, kp, vp, tab, lens = (prob[x] for x in ("q", "k_pages", "v_pages", "block_table", "seq_lens"))
        B, Hq, d = q.shape
        H = kp.shape[1]
        G = Hq // H
        sc = 0.3
        res = OB.blocktopk_decode(q, kp, vp, tab, lens, sc, k, store="f32")
        for b in range(B):
            L = int(lens[b])
            nb = (L + 15) // 16
            for h in range(H):
                keys = np.concatenate([kp[tab[b, j], h] for j in range(nb)]).astype(np.float64)
                vals = np.concatenate([vp[tab[b, j], h] for j in range(nb)]).astype(np.float64)
                cent = keys[: 16 * (nb - 1)].reshape(nb - 1, 16, d).mean(axis=1)
                qg = q[b, h * G:(h + 1) * G].astype(np.float64)
                s = cent @ qg.sum(axis=0)
                sel = _brute_force_select(list(s), nb, k)
                assert list(res["sel"][b, h, :len(sel)]) == sel
                mask = torch.zeros(16 * nb, dtype=torch.bool)
                for j in sel:
                    mask[16 * j: 16 * j + 16] = True
                mask[L:] = False
                ref = torch.nn.functional.scaled_dot_product_attention(
                    torch.tensor(qg)[None, :, None, :],
                    torch.tensor(keys)[None, None].expand(1, G, -1, d),
                    torch.tensor(vals)[None, None].expand(1, G, -1, d),
                    attn_mask=mask[None, None, None, :], scale=sc)[0, :, 0, :].numpy()
                assert np.allclose(res["out"][b, h * G:(h + 1) * G], ref, rtol=1e-10, atol=1e-12)
                assert np.allclose(res["scores"][b, h, :nb - 1], s, rtol=1e-5, atol=1e-6)


def pin_decode_invariants():
    prob, k = _tiny_problem(30)
    args = (prob["q"], prob["k_pages"], prob["v_pages"], prob["block_table"], prob["seq_lens"], 0.25)
    base = OB.blocktopk_decode(*args, k, store="bf16")
    # k >= number of blocks: block top-k is dense decode, bit for bit
    big = OB.blocktopk_decode(*args, 64, store="bf16")
    dense = OB.dense_decode(*args)
    assert np.array_equal(big["out"], dense["out"]) and np.array_equal(big["lse"], dense["lse"])
    # a positive scale of q changes no selection
    scaled = OB.blocktopk_decode(prob["q"] * 3.5, *args[1:], k, store="bf16")
    assert np.array_equal(scaled["sel"], base["sel"])
    # physical page placement does not matter
    P = prob["k_pages"].shape[0]
    perm = _rng(31).permutation(P)
    inv = np.argsort(perm)
    tab2 = np.where(prob["block_table"] >= 0, inv[np.maximum(prob["block_table"], 0)], -1)
    moved = OB.blocktopk_decode(prob["q"], prob["k_pages"][perm], prob["v_pages"][perm], tab2,
                                prob["seq_lens"], 0.25, k, store="bf16")
    for key in ("out", "lse", "sel"):
        assert np.array_equal(moved[key], base[key])
    # stale slots past the length are never read
    kp2, vp2 = prob["k_pages"].copy(), prob["v_pages"].copy()
    for b, L in enumerate(prob["seq_lens"]):
        nb = (int(L) + 15) // 16
        p = prob["block_table"][b, nb - 1]
        kp2[p, :, int(L) - 16 * (nb - 1):] = -7.0
        vp2[p, :, int(L) - 16 * (nb - 1):] = 9.0
    st = OB.blocktopk_decode(prob["q"], kp2, vp2, *args[3:], k, store="bf16")
    assert np.array_equal(st["out"], base["out"])
    # duplicating a block's keys into a later block: the lower index wins the tie
    kp3 = prob["k_pages"].copy()
    tab = prob["block_table"]
    kp3[tab[1, 4]] = kp3[tab[1, 1]]
    dup = OB.blocktopk_decode(prob["q"], kp3, *args[2:], 2, store="bf16")
    for h in range(kp3.shape[1]):
        s = dup["scores"][1, h]
        assert s[1] == s[4]
        if int(np.argmax(s[:6])) in (1, 4):
            assert list(dup["sel"][1, h]) == [1, 6]


def pin_hand_worked_golden():
    g = json.load(open(os.path.join(GOLDEN, "hand_worked_tiny.json")))
    ev = lambda e: eval(e, {"sqrt": math.sqrt, "log": math.log})  # closed forms only
    k_pages = np.full((3, 1, 16, 2), 1e3, dtype=np.float32)
    v_pages = np.full((3, 1, 16, 2), -1e3, dtype=np.float32)
    for t in range(16):
        k_pages[2, 0, t] = (1.0, 0.0) if t % 2 == 0 else (3.0, 0.0)
        v_pages[2, 0, t] = (1.0, 0.0) if t % 2 == 0 else (0.0, 1.0)
        k_pages[0, 0, t] = (0.0, 1.0) if t % 2 == 0 else (0.0, 3.0)
        v_pages[0, 0, t] = (-1.0, 0.0)
    k_pages[1, 0, :8] = (0.5, 0.5)
    v_pages[1, 0, :8] = (1.0, 1.0)
    q = np.array(g["q"], dtype=np.float32)[None]
    tab = np.array([g["block_table"]])
    lens = np.array([g["seq_len"]])
    sc = math.log(2.0)
    sp = OB.blocktopk_decode(q, k_pages, v_pages, tab, lens, sc, g["top_k"], store="f32")
    de = OB.dense_decode(q, k_pages, v_pages, tab, lens, sc)
    e = g["expected"]
    assert list(sp["scores"][0, 0, :2]) == [ev(x) for x in e["scores"]]
    assert list(sp["sel"][0, 0]) == e["selection"]
    for key, res in (("sparse", sp), ("dense", de)):
        want_o = np.array([[ev(x) for x in row] for row in e[key + "_out"]])
        want_l = np.array([ev(x) for x in e[key + "_lse"]])
        assert np.allclose(res["out"][0], want_o, rtol=1e-13, atol=1e-14)
        assert np.allclose(res["lse"][0], want_l, rtol=1e-13, atol=1e-14)


# ----------------------------------------------------------------------------- bytes
def pin_byte_accounting():
    g = json.load(open(os.path.join(GOLDEN, "cost_model_units.json")))
    kv = g["kv_cache_per_sequence"]
    sh = kv["shape_used"]
    per_layer = OB.dense_kv_bytes_per_step(kv["tokens"], sh["num_kv_heads"], sh["head_dim"],
                                           sh["bytes_per_element"])
    assert per_layer * sh["layers"] == kv["kv_bytes"]
    # dense decode over L_out generated tokens: sum of per-step reads = D * L_out * (L_out + 1)
    for H, d in ((8, 128), (1, 64)):
        D = 2 * H * d
        for Lout in (1, 16, 1000, 4097):
            tot = sum(OB.dense_kv_bytes_per_step(L, H, d, 2) for L in range(1, Lout + 1))
            assert tot == D * Lout * (Lout + 1)
    # sparse: at most B = k * 16 tokens per step, exactly B when the final block is full
    bf = g["benchmark_flags"]
    k = bf["topk_page"]
    assert k * bf["page_size"] == bf["token_budget"]
    for L in range(1, 4 * k * 16):
        T = OB.sparse_kv_tokens(L, k)
        nb = (L + 15) // 16
        if nb <= k:
            assert T == L
        else:
            assert (k - 1) * 16 < T <= k * 16
            if L % 16 == 0:
                assert T == bf["token_budget"]
    # decode_bytes counts exactly the tokens the oracle gathers, plus scored centroids
    prob, kk = _tiny_problem(40)
    res = OB.blocktopk_decode(prob["q"], prob["k_pages"], prob["v_pages"], prob["block_table"],
                              prob["seq_lens"], 0.1, kk, store="f32")
    H, d = prob["k_pages"].shape[1], prob["k_pages"].shape[3]
    G = prob["q"].shape[1] // H
    toks = 0
    for b, L in enumerate(prob["seq_lens"]):
        for h in range(H):
            for j in res["sel"][b, h]:
                if j >= 0:
                    toks += min(16, int(L) - 16 * int(j))
    nbs = [(int(L) + 15) // 16 for L in prob["seq_lens"]]
    byt = OB.decode_bytes(prob["seq_lens"], H, G, d, kk, 4)
    assert byt["kv"] == 2 * toks * d * 4
    assert byt["centroids"] == sum((n - 1) * H * d * 4 for n in nbs if n > kk)
    assert byt["qo"] == 2 * len(nbs) * H * G * d * 4


PINS = [pin_bf16_rounding, pin_centroid_closed_forms, pin_centroid_pair, pin_group_scores,
        pin_valid_selections,
        pin_selection_brute_force, pin_attention_vs_sdpa, pin_decode_against_masked_sdpa,
        pin_decode_invariants, pin_hand_worked_golden, pin_byte_accounting]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ----------------------------------------------------------------------------- mutants
def _m_no_forced_final(scores, nb, k):
    if nb <= k:
        return list(range(nb))
    order = sorted(range(nb - 1), key=lambda j: (-float(scores[j]), j))
    return sorted(order[:k])


def _m_ties_high(scores, nb, k):
    if nb <= k:
        return list(range(nb))
    order = sorted(range(nb - 1), key=lambda j: (-float(scores[j]), -j))
    return sorted(order[: k - 1] + [nb - 1])


def _m_lowest(scores, nb, k):
    if nb <= k:
        return list(range(nb))
    order = sorted(range(nb - 1), key=lambda j: (float(scores[j]), j))
    return sorted(order[: k - 1] + [nb - 1])


def _m_extra_block(scores, nb, k):
    if nb <= k:
        return list(range(nb))
    order = sorted(range(nb - 1), key=lambda j: (-float(scores[j]), j))
    return sorted(order[:k] + [nb - 1])


def _m_first_head_only(q_group, cents):
    return np.asarray(cents, np.float64) @ np.asarray(q_group, np.float64)[0]


def _m_no_length_mask(k_pages, v_pages, table_row, seq_len, blocks, h):
    ks = [np.asarray(k_pages[int(table_row[j]), h], np.float64) for j in blocks]
    vs = [np.asarray(v_pages[int(table_row[j]), h], np.float64) for j in blocks]
    return np.concatenate(ks), np.concatenate(vs)


def _m_no_scale(q_group, keys, vals, sm_scale):
    return _orig_attend(q_group, keys, vals, 1.0)


def _m_lse_no_max(q_group, keys, vals, sm_scale):
    o, lse = _orig_attend(q_group, keys, vals, sm_scale)
    z = sm_scale * (np.asarray(q_group, np.float64) @ np.asarray(keys, np.float64).T)
    return o, lse - z.max(axis=1)


def _m_centroid_div15(keys, store="f32"):
    acc = np.asarray(keys, np.float32).sum(axis=0, dtype=np.float32)
    return OB._store((acc / np.float32(15.0)).astype(np.float32), store)


def _m_centroids_wrong_axis(k_pages, page_ids, store):
    blk = np.asarray(k_pages[np.asarray(page_ids)], dtype=np.float32)
    return OB._store(blk.mean(axis=3, keepdims=True).repeat(blk.shape[3], 3)[:, :, 0, :], store)


def _m_bf16_truncate(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)


def _m_pair_no_residual(k_pages, page_ids):
    hi, lo = _orig_pair(k_pages, page_ids)
    return hi, np.zeros_like(lo)


def _m_pair_residual_sign(k_pages, page_ids):
    hi, lo = _orig_pair(k_pages, page_ids)
    return hi, -lo


def _m_valid_absolute_band(scores, nb, k, rel=1e-3, limit=100000):
    # the band taken in absolute units instead of relative to the last kept score
    base = OB.select_blocks(scores, nb, k)
    if nb <= k or k == 1:
        return [base]
    cand = [float(scores[j]) for j in range(nb - 1)]
    t = sorted(cand, reverse=True)[k - 2]
    near = [j for j in range(nb - 1) if abs(cand[j] - t) <= rel]
    core = [j for j in base[:-1] if j not in near]
    return [sorted(core + list(c) + [nb - 1])
            for c in itertools.combinations(near, k - 1 - len(core))]


def _m_valid_only_base(scores, nb, k, rel=1e-3, limit=100000):
    return [OB.select_blocks(scores, nb, k)]


_orig_pair = OB.centroid_pair
_orig_attend = OB.attend

MUTANTS = {
    "no_forced_final_block": ("select_blocks", _m_no_forced_final),
    "ties_to_higher_index": ("select_blocks", _m_ties_high),
    "lowest_scores_kept": ("select_blocks", _m_lowest),
    "k_plus_one_blocks": ("select_blocks", _m_extra_block),
    "score_first_head_only": ("group_scores", _m_first_head_only),
    "stale_slots_read": ("row_tokens", _m_no_length_mask),
    "softmax_scale_dropped": ("attend", _m_no_scale),
    "lse_missing_max": ("attend", _m_lse_no_max),
    "centroid_divides_by_15": ("block_centroid", _m_centroid_div15),
    "centroid_wrong_axis": ("centroids", _m_centroids_wrong_axis),
    "bf16_truncates": ("round_to_bf16", _m_bf16_truncate),
    "pair_without_residual": ("centroid_pair", _m_pair_no_residual),
    "pair_residual_wrong_sign": ("centroid_pair", _m_pair_residual_sign),
    "admissible_band_absolute": ("valid_selections", _m_valid_absolute_band),
    "admissible_only_own_set": ("valid_selections", _m_valid_only_base),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(OB, attr, fn)
    failed = []
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
        except Exception:          # a crash elsewhere is not what we look for
            pass
    assert failed, f"no pin caught the planted mistake {name}"
