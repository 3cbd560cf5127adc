"""Pins of the token-level top-k oracle (``oracle.tokentopk``) against things other than
itself (CPU only): closed forms, brute-force enumeration of kept sets, torch's scaled dot
product attention over a mask, the dense decode oracle, and the block top-k oracle on
keys that are constant within each block.  The mutation tests at the end plant plausible
mistakes and check that a pin fails for each.
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle.blocktopk as OB
import oracle.tokentopk as OT


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16_exact(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy()


# ----------------------------------------------------------------------------- scores
def pin_token_scores_closed_form():
    """s_t = sum_g q_g . k_t: integer inputs against the exact rational sum, and a
    one-hot closed form."""
    G, d, T = 3, 8, 11
    q = np.zeros((G, d), np.float32)
    for g in range(G):
        q[g, g] = g + 1.0                      # q_g = (g + 1) e_g
    k = np.array([[10.0 * t + i for i in range(d)] for t in range(T)], np.float32)
    want = [sum((g + 1) * (10 * t + g) for g in range(G)) for t in range(T)]
    assert np.array_equal(OT.token_scores(q, k), np.array(want, np.float64))
    r = _rng(3)
    q = r.integers(-9, 10, (4, 16)).astype(np.float32)
    k = r.integers(-9, 10, (30, 16)).astype(np.float32)
    exact = [sum(Fraction(int(q[g, i])) * int(k[t, i]) for g in range(4) for i in range(16))
             for t in range(30)]
    assert [Fraction(float(s)) for s in OT.token_scores(q, k)] == exact


# ----------------------------------------------------------------------------- select
def _brute_top(scores, budget):
    """The kept set by enumeration: the budget-subset with the largest score sum (distinct
    scores make it unique)."""
    n = len(scores)
    if n <= budget:
        return list(range(n))
    best = max(itertools.combinations(range(n), budget),
               key=lambda c: sum(Fraction(float(scores[t])) for t in c))
    return sorted(best)


def pin_select_tokens():
    r = _rng(4)
    for _ in range(300):
        n = int(r.integers(1, 10))
        budget = int(r.integers(1, n + 2))
        s = r.permutation(n).astype(np.float64) + r.standard_normal() * 1e-3
        assert OT.select_tokens(s, budget) == _brute_top(s, budget)
    # ties go to the lower position (reading T4); no position is forced in (T3)
    assert OT.select_tokens([5.0] * 7, 3) == [0, 1, 2]
    assert OT.select_tokens([1.0, 2.0, 2.0, 2.0, 0.0], 2) == [1, 2]
    assert OT.select_tokens([3.0, 1.0, 2.0, 0.0], 2) == [0, 2]
    assert OT.select_tokens([1.0, 2.0], 5) == [0, 1]


def pin_token_admissible():
    s = [9.0, 1.0, 5.0, 4.999, 3.0, 5.0002, 0.5]
    budget = 3                                 # oracle keeps 0, 2, 5; B-th score 5.0
    assert OT.token_admissible(s, [0, 2, 5], budget, 1e-2)
    assert OT.token_admissible(s, [0, 3, 5], budget, 1e-2)        # 4.999 within 0.01
    assert OT.token_admissible(s, [5, 0, 3], budget, 1e-2)        # order does not matter
    assert not OT.token_admissible(s, [0, 3, 5], budget, 1e-4)    # not within 1e-4
    assert not OT.token_admissible(s, [0, 2, 4], budget, 1e-2)    # 3.0 is far below
    assert not OT.token_admissible(s, [0, 2], budget, 1e-2)       # too few
    assert not OT.token_admissible(s, [0, 2, 2], budget, 1e-2)    # repeated
    assert not OT.token_admissible(s, [0, 2, 7], budget, 1e-2)    # outside the row
    assert OT.token_admissible([1.0, 2.0], [0, 1], 4, 0.0)        # short row: all
    assert not OT.token_admissible([1.0, 2.0], [1], 4, 10.0)


# ----------------------------------------------------------------------------- decode
def _tiny(seed, B=2, H=2, G=2, d=16, lens=(37, 70), const_blocks=False):
    r = _rng(seed)
    maxb = max((L + 15) // 16 for L in lens)
    P = B * maxb + 3
    k = _bf16_exact(r.standard_normal((P, H, 16, d)))
    if const_blocks:
        k = np.repeat(k[:, :, :1, :], 16, axis=2)
    v = _bf16_exact(r.standard_normal((P, H, 16, d)))
    q = _bf16_exact(r.standard_normal((B, H * G, d)))
    table = r.permutation(P)[:B * maxb].reshape(B, maxb).astype(np.int64)
    return q, k, v, table, np.array(lens, np.int64)


def pin_token_against_masked_sdpa():
    """Kept set by enumeration of exact score sums and attention by torch's scaled dot
    product attention over that mask, against the oracle's output."""
    q, k, v, table, lens = _tiny(5, lens=(9, 7), d=8)
    budget, scale = 4, 0.7
    res = OT.tokentopk_decode(q, k, v, table, lens, scale, budget)
    B, Hq, d = q.shape
    H = k.shape[1]
    G = Hq // H
    for b in range(B):
        L = int(lens[b])
        for h in range(H):
            keys = np.stack([k[table[b, t // 16], h, t % 16] for t in range(L)]).astype(np.float64)
            vals = np.stack([v[table[b, t // 16], h, t % 16] for t in range(L)]).astype(np.float64)
            qg = q[b, h * G:(h + 1) * G].astype(np.float64)
            s = [sum(Fraction(float(qg[g, i])) * Fraction(float(keys[t, i]))
                     for g in range(G) for i in range(d)) for t in range(L)]
            kept = _brute_top([float(x) for x in s], budget)
            assert list(res["sel"][b, h, :len(kept)]) == kept
            mask = torch.zeros(1, L, dtype=torch.bool)
            mask[0, kept] = True
            o = torch.nn.functional.scaled_dot_product_attention(
                torch.tensor(qg)[None], torch.tensor(keys)[None], torch.tensor(vals)[None],
                attn_mask=mask[None], scale=scale)[0].numpy()
            assert np.allclose(res["out"][b, h * G:(h + 1) * G], o, atol=1e-12, rtol=1e-10)


def pin_token_dense_when_budget_covers_row():
    """B >= L keeps every token: the output is the dense decode oracle's, bit for bit."""
    q, k, v, table, lens = _tiny(6, lens=(37, 70))
    t = OT.tokentopk_decode(q, k, v, table, lens, 0.25, 80)
    dd = OB.dense_decode(q, k, v, table, lens, 0.25)
    assert np.array_equal(t["out"], dd["out"]) and np.array_equal(t["lse"], dd["lse"])
    assert list(t["sel"][1, 0, :70]) == list(range(70)) and t["sel"][1, 0, 70] == -1


def pin_token_equals_block_on_block_constant_keys():
    """Keys constant within each block: a block's fp32 centroid is its key exactly, so block
    scores equal token scores.  With full blocks, distinct block scores and the final block
    scoring highest (so that block top-k's forced final block is also a top block), token
    top-16k keeps exactly the tokens of block top-k's k blocks, and the outputs agree bit
    for bit (same tokens, same order)."""
    q, k, v, table, lens = _tiny(7, lens=(64, 96), const_blocks=True)
    B, Hq, d = q.shape
    H = k.shape[1]
    G = Hq // H
    for b in range(B):
        nb = int(lens[b]) // 16
        for h in range(H):
            qs = q[b, h * G:(h + 1) * G].sum(axis=0)
            k[table[b, nb - 1], h] = _bf16_exact(np.repeat(4.0 * qs[None] / np.abs(qs).max(), 16, 0))
    kk = 3
    blk = OB.blocktopk_decode(q, k, v, table, lens, 0.3, kk, store="f32")
    tok = OT.tokentopk_decode(q, k, v, table, lens, 0.3, 16 * kk)
    for b in range(B):
        for h in range(H):
            blocks = [int(j) for j in blk["sel"][b, h] if j >= 0]
            assert len(blocks) == kk and blocks[-1] == int(lens[b]) // 16 - 1
            want = [16 * j + t for j in blocks for t in range(16)]
            assert list(tok["sel"][b, h]) == want
    assert np.array_equal(tok["out"], blk["out"]) and np.array_equal(tok["lse"], blk["lse"])


def pin_token_bytes():
    byt = OT.token_decode_bytes([37, 70], 2, 3, 16, 40, 2)
    assert byt["all_k"] == (37 + 70) * 2 * 16 * 2
    assert byt["kept_kv"] == (37 + 40) * 2 * 2 * 16 * 2
    assert byt["qo"] == 2 * 2 * 2 * 3 * 16 * 2
    assert byt["total"] == byt["all_k"] + byt["kept_kv"] + byt["qo"]


PINS = [pin_token_scores_closed_form, pin_select_tokens, pin_token_admissible,
        pin_token_against_masked_sdpa, pin_token_dense_when_budget_covers_row,
        pin_token_equals_block_on_block_constant_keys, pin_token_bytes]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_token_pin(pin):
    pin()


# ----------------------------------------------------------------------------- mutants
_orig_select = OT.select_tokens
_orig_admissible = OT.token_admissible


def _m_first_head(q_group, keys):
    return np.asarray(keys, np.float64) @ np.asarray(q_group, np.float64)[0]


def _m_ties_high(scores, budget):
    n = len(scores)
    if n <= budget:
        return list(range(n))
    return sorted(sorted(range(n), key=lambda t: (-float(scores[t]), -t))[:budget])


def _m_lowest(scores, budget):
    n = len(scores)
    if n <= budget:
        return list(range(n))
    return sorted(sorted(range(n), key=lambda t: (float(scores[t]), t))[:budget])


def _m_force_current(scores, budget):
    n = len(scores)
    if n <= budget:
        return list(range(n))
    order = [t for t in sorted(range(n), key=lambda t: (-float(scores[t]), t)) if t != n - 1]
    return sorted(order[:budget - 1] + [n - 1])


def _m_one_extra(scores, budget):
    return _orig_select(scores, budget + 1)


def _m_keep_all(scores, budget):
    return list(range(len(scores)))


def _m_admit_all(scores, kept, budget, tol):
    return True


def _m_admit_only_own(scores, kept, budget, tol):
    return sorted(int(t) for t in kept) == _orig_select(scores, budget)


MUTANTS = {
    "token_score_first_head_only": ("token_scores", _m_first_head),
    "token_ties_to_higher_position": ("select_tokens", _m_ties_high),
    "token_lowest_scores_kept": ("select_tokens", _m_lowest),
    "token_current_forced_in": ("select_tokens", _m_force_current),
    "token_budget_plus_one": ("select_tokens", _m_one_extra),
    "token_selection_ignored": ("select_tokens", _m_keep_all),
    "token_admits_anything": ("token_admissible", _m_admit_all),
    "token_admits_only_own_set": ("token_admissible", _m_admit_only_own),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_token_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(OT, attr, fn)
    failed = []
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
        except Exception:          # a crash elsewhere is not what we look for
            pass
    assert failed, f"no pin caught the planted mistake {name}"
