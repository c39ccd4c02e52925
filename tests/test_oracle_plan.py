"""Pins of the oracle's rounding, gating and permutation (CPU only).

Each check compares the oracle with something other than itself: a library
routine, a brute force, a closed form, or a hand-worked fixture.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle.moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- rounding
def test_bf16_round_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    a = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        rng.standard_normal(1000) * 1e-39]).astype(np.float32)
    ref = torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.bf16_round(a.astype(np.float64)), ref)


def test_bf16_round_special_cases():
    u = 2.0 ** -7  # spacing of bf16 just above 1
    cases = {
        1.0 + u / 2: 1.0,                 # tie -> even mantissa
        1.0 + 3 * u / 2: 1.0 + 2 * u,     # tie -> even mantissa (upwards)
        1.0 + u / 2 + 1e-12: 1.0 + u,     # just above the tie
        -(1.0 + u / 2): -1.0,
        2.0 ** -133: 2.0 ** -133,         # smallest subnormal
        2.0 ** -134: 0.0,                 # tie between 0 and it -> 0
        1.5 * 2.0 ** -133: 2.0 ** -132,   # tie -> even
        3.3962e38: math.inf,              # above max + half ulp (3.39618e38)
        3.3961e38: 3.3895313892515355e38, # below it: rounds to the largest finite
        3.3895e38: 3.3895313892515355e38,
    }
    for a, b in cases.items():
        assert O.bf16_round(np.array([a]))[0] == b, a
    assert np.isnan(O.bf16_round(np.array([np.nan]))[0])


# ---------------------------------------------------------------- gating
def _brute_topk(l, k):
    out = []
    for row in l.tolist():
        order = sorted(range(len(row)), key=lambda e: (-row[e], e))
        out.append(order[:k])
    return np.array(out)


@pytest.mark.parametrize("T,E,k", [(64, 8, 2), (40, 16, 5), (33, 6, 6), (17, 5, 1)])
def test_topk_matches_brute_force_with_ties(T, E, k):
    rng = np.random.default_rng(T * E + k)
    l = rng.integers(-3, 3, size=(T, E)).astype(np.float32)  # many ties
    l[::3] = rng.standard_normal((len(l[::3]), E)).astype(np.float32)
    ids, w = O.route(l, k)
    assert np.array_equal(ids, _brute_topk(l, k))


def test_weights_equal_softmax_then_renormalise():
    rng = np.random.default_rng(1)
    l = (rng.standard_normal((200, 32)) * 3).astype(np.float32)
    ids, w = O.route(l, 6)
    p = np.exp(l.astype(np.float64))
    p /= p.sum(axis=1, keepdims=True)           # softmax over all E
    top = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    lit = top / top.sum(axis=1, keepdims=True)  # renormalise over the k
    assert np.allclose(w, lit, rtol=2e-7, atol=0)
    assert np.all(np.abs(w.astype(np.float64).sum(axis=1) - 1.0) <= 6 * 2.0 ** -24)


def test_weights_closed_forms():
    rng = np.random.default_rng(2)
    l = rng.standard_normal((50, 7)).astype(np.float32)
    ids, w = O.route(l, 1)
    assert np.all(w == 1.0)
    ids, w = O.route(l, 7)  # k = E: the full softmax, experts in descending order
    p = np.exp(l.astype(np.float64) - l.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    assert np.allclose(w, np.take_along_axis(p, ids.astype(np.int64), 1), rtol=2e-7)
    assert np.all(np.diff(w, axis=1) <= 0)


def test_nonfinite_logit_rejected():
    l = np.zeros((4, 4), np.float32)
    l[2, 1] = np.nan
    with pytest.raises(ValueError):
        O.route(l, 2)


# ---------------------------------------------------------------- permutation
def test_hand_worked_fixture():
    g = json.load(open(os.path.join(GOLDEN, "permutation_tiny.json")))
    l = np.array(g["logits"], np.float32)
    ids, w = O.route(l, g["k"])
    assert ids.tolist() == g["ids"]
    for t, d in enumerate(g["weight_gap"]):
        s = 1.0 / (1.0 + math.exp(-d))
        assert w[t, 0] == np.float32(s) and abs(w[t, 1] - (1 - s)) <= 2 ** -24
    p = O.permutation(ids, g["E"])
    assert p.counts.tolist() == g["counts"]
    assert p.offsets.tolist() == g["offsets"]
    assert p.dest.tolist() == g["dest"]
    assert p.row_src.tolist() == g["row_src"]
    assert p.row_slot.tolist() == g["row_slot"]


def _random_ids(T, E, k, seed, skew=0.0):
    rng = np.random.default_rng(seed)
    l = rng.standard_normal((T, E)).astype(np.float32)
    l += (skew * np.log(np.arange(1, E + 1) ** -1.2)).astype(np.float32)
    return O.route(l, k)[0]


@pytest.mark.parametrize("T,E,k,skew", [(256, 8, 2, 0), (300, 13, 4, 3.0), (1, 5, 3, 0), (97, 64, 6, 8.0)])
def test_permutation_is_stable_sort(T, E, k, skew):
    ids = _random_ids(T, E, k, T + E, skew)
    p = O.permutation(ids, E)
    flat = ids.reshape(-1).astype(np.int64)
    order = np.argsort(flat, kind="stable")       # library stable sort of the pairs
    assert np.array_equal(p.row_src, order // k)
    assert np.array_equal(p.row_slot, order % k)
    assert np.array_equal(p.counts, np.bincount(flat, minlength=E))
    # invariants
    R = T * k
    assert p.counts.sum() == R and p.offsets[0] == 0 and p.offsets[-1] == R
    for e in range(E):
        seg = p.row_src[p.offsets[e]:p.offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)           # strictly increasing token ids
    assert sorted(p.dest.reshape(-1).tolist()) == list(range(R))  # bijection
    for t in range(T):
        for j in range(k):
            r = p.dest[t, j]
            e = ids[t, j]
            assert p.offsets[e] <= r < p.offsets[e + 1]
            assert p.row_src[r] == t and p.row_slot[r] == j


def test_permutation_closed_form_E_equals_k():
    T, E = 37, 5
    ids = _random_ids(T, E, E, 3)
    p = O.permutation(ids, E)
    assert np.all(p.counts == T)
    for t in range(T):
        for j in range(E):
            assert p.dest[t, j] == p.offsets[ids[t, j]] + t


def test_unpermute_after_permute_is_identity():
    T, E, k, H = 50, 6, 3, 8
    ids = _random_ids(T, E, k, 4)
    p = O.permutation(ids, E)
    x = np.random.default_rng(5).standard_normal((T, H))
    Xp = O.gather(x, p.row_src)
    for j in range(k):
        assert np.array_equal(Xp[p.dest[:, j]], x)
    assert np.array_equal(O.unpermute_sum(Xp, p.dest, mirror=False), k * x)


def test_empty_experts():
    ids = np.array([[0, 3], [3, 0], [0, 3]], np.int32)
    p = O.permutation(ids, 6)
    assert p.counts.tolist() == [3, 0, 0, 3, 0, 0]
    assert p.offsets.tolist() == [0, 3, 3, 3, 6, 6, 6]
