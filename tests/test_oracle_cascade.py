"""Pins of the LAVa online-prefill cascade oracle against what the LAVa page and the
mathematics fix, independently of the cascade's own code:

- with caps that cannot bind, the capped split is the one-shot LAVa layer split
  (lava_layer_budgets, itself pinned in test_oracle_pins);
- the whole budget is in use after every stage (sum of layer budgets = total), each layer's
  budget only shrinks from stage to stage, and the rows a layer keeps are nested;
- choosing among the rows a layer still holds gives what choosing among all its candidates
  gives (top-B sets of one total order are nested), computed with Algorithm 1's counts and
  the per-head Top-k, not with the cascade's selection;
- when the caps never bind, the last stage is the one-shot LAVa eviction: its budgets and
  kept sets equal lava_layer_budgets / head_budgets(alpha = 0) / topk_positions;
- peak memory: the rows held when layer t-1 has been prefilled are the earlier layers'
  budgets (at most the total) plus n*Hkv, against L*n*Hkv for a prefill of every layer
  before eviction;
- a hand-derived case of identical layers.
"""
import numpy as np
import pytest

import oracle as O


def rand_layers(rng, L, hkv, C, spread):
    S = []
    for _ in range(L):
        temp = np.exp(rng.uniform(-1, 1) * spread)
        x = rng.gamma(0.3, size=(hkv, C)) ** temp
        S.append(x / x.sum())
    return S


@pytest.mark.parametrize("seed", range(6))
def test_uncapped_split_is_the_one_shot_lava_split(seed):
    rng = np.random.default_rng(seed)
    L, hkv, C, w = 5, 3, 40, 2
    e = rng.random(L) * (rng.random(L) > 0.2)
    total = int(rng.integers(L * w * hkv, L * (w * hkv + hkv * C)))
    ref = O.lava_layer_budgets(e, total, w, hkv, C) - w * hkv
    got = O.capped_split(e, total - L * w * hkv, [hkv * C] * L)
    np.testing.assert_array_equal(got, ref)


def test_capped_split_respects_caps_and_sums():
    rng = np.random.default_rng(7)
    for _ in range(200):
        L = int(rng.integers(1, 7))
        e = rng.random(L)
        caps = rng.integers(0, 50, L)
        R = int(rng.integers(0, caps.sum() + 1))
        s = O.capped_split(e, R, caps)
        assert s.sum() == R
        assert np.all(s <= caps) and np.all(s >= 0)


@pytest.mark.parametrize("seed", range(8))
def test_cascade_stages(seed):
    rng = np.random.default_rng(100 + seed)
    L, hkv, C, w = 5, 2, 30, 3
    n = C + w
    S = rand_layers(rng, L, hkv, C, spread=2.0)
    total = int(rng.integers(L * w * hkv + 4, L * w * hkv + 2 * hkv * C))
    st = O.lava_cascade(S, total, w, n)
    assert len(st) == L
    prev = None
    for t, x in enumerate(st, start=1):
        lb, hb = x["layer_budget"], x["head_budget"]
        # the whole budget in use at every stage, unless the layers so far hold less
        held = n * hkv + (0 if prev is None else int(prev["layer_budget"].sum()))
        assert len(lb) == t and lb.sum() == min(total, held)
        np.testing.assert_array_equal(hb.sum(axis=1), lb)
        assert x["rows_after"] == lb.sum()
        assert x["rows_before"] == held
        for l in range(t):
            for g in range(hkv):
                kept = x["kept"][l][g]
                assert len(kept) == hb[l, g]
                assert np.all(np.diff(kept) > 0) and np.all(kept[-w:] == np.arange(C, n))
            # the held-rows choice equals Algorithm 1 over every candidate of the layer
            Bp = int(lb[l]) - w * hkv
            f = O.global_topk_counts(S[l], Bp)
            np.testing.assert_array_equal(hb[l] - w, f)
            for g in range(hkv):
                np.testing.assert_array_equal(x["kept"][l][g][:-w], O.topk_positions(S[l][g],
                                                                                     int(f[g])))
        if prev is not None:
            assert np.all(lb[:-1] <= prev["layer_budget"])     # budgets only shrink
            for l in range(t - 1):
                for g in range(hkv):
                    assert set(x["kept"][l][g]) <= set(prev["kept"][l][g])   # nested
        prev = x


def test_last_stage_is_the_one_shot_eviction_when_caps_never_bind():
    rng = np.random.default_rng(11)
    L, hkv, C, w = 6, 2, 50, 2
    n = C + w
    checked = 0
    for _ in range(40):
        S = rand_layers(rng, L, hkv, C, spread=1.0)
        total = int(rng.integers(L * w * hkv + 10, L * w * hkv + hkv * C))
        st = O.lava_cascade(S, total, w, n)
        if any(x["caps_bound"] for x in st):
            continue
        checked += 1
        e = [O.layer_entropy(S[l], n) for l in range(L)]
        lb = O.lava_layer_budgets(e, total, w, hkv, C)
        last = st[-1]
        np.testing.assert_array_equal(last["layer_budget"], lb)
        for l in range(L):
            f, Bg = O.head_budgets(S[l], int(lb[l]), w, 0, 1)
            np.testing.assert_array_equal(last["head_budget"][l], Bg + w)
            for g in range(hkv):
                np.testing.assert_array_equal(last["kept"][l][g][:-w],
                                              O.topk_positions(S[l][g], int(Bg[g])))
    assert checked >= 10


def test_identical_layers_hand_derived():
    """Three identical layers, one KV head, C = 4, w = 1, total 9 (window rows included).
    Equal entropies: stage 1 gives layer 0 all 9 - 1 = 8 selectable rows, capped at C = 4;
    stage 2 shares 9 - 2 = 7 as 3.5 / 3.5 -> floors 3, 3, one remainder unit to the lower
    layer: (4, 3); stage 3 shares 6 as 2, 2, 2.  Scores 0.4, 0.1, 0.3, 0.2 keep positions
    {0, 2} once two remain, {0, 2, 3} with three."""
    s = np.array([[0.4, 0.1, 0.3, 0.2]])
    st = O.lava_cascade([s, s, s], total=9, w=1, n=5)
    np.testing.assert_array_equal(st[0]["layer_budget"], [5])
    np.testing.assert_array_equal(st[1]["layer_budget"], [5, 4])
    np.testing.assert_array_equal(st[2]["layer_budget"], [3, 3, 3])
    np.testing.assert_array_equal(st[1]["kept"][1][0], [0, 2, 3, 4])
    for l in range(3):
        np.testing.assert_array_equal(st[2]["kept"][l][0], [0, 2, 4])
