"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Nothing here runs the CUDA path.  Each test ties one oracle function to an
independent fact: a closed form, a brute-force optimum, one of the pages'
theorems, or a special case that reduces to a library routine (torch's
max_pool1d and scaled_dot_product_attention in fp64).
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle as O

RNG = np.random.default_rng(1234)


# --------------------------------------------------------------------------
# Window attention (Ada-KV Algorithm 2, first step; LaProx Eq. 2 scale)
# --------------------------------------------------------------------------

def test_window_attention_equal_logits_closed_form():
    """q = 0: every visible key gets 1/(number visible); row t sees n-w+t+1 keys."""
    hq, hkv, w, n, d = 4, 2, 5, 23, 8
    q = np.zeros((hq, w, d))
    k = RNG.normal(size=(hkv, n, d))
    P = O.window_attention(q, k, scale=0.3)
    for t in range(w):
        vis = n - w + t + 1
        np.testing.assert_allclose(P[:, t, :vis], 1.0 / vis, rtol=0, atol=1e-15)
        assert np.all(P[:, t, vis:] == 0.0)


def test_window_attention_matches_sdpa_weights():
    """SDPA with V = identity returns the attention weights themselves."""
    hq, hkv, w, n, d = 6, 2, 7, 40, 16
    q = RNG.normal(size=(hq, w, d)) * 2.0
    k = RNG.normal(size=(hkv, n, d))
    scale = 1.0 / math.sqrt(d)
    P = O.window_attention(q, k, scale)
    G = hq // hkv
    mask = torch.zeros(w, n, dtype=torch.bool)
    for t in range(w):
        mask[t, : n - w + t + 1] = True
    eye = torch.eye(n, dtype=torch.float64)
    for qh in range(hq):
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[qh])[None], torch.from_numpy(k[qh // G])[None], eye[None],
            attn_mask=mask[None], scale=scale)[0].numpy()
        np.testing.assert_allclose(P[qh], ref, rtol=1e-12, atol=1e-15)


def test_window_attention_prefix_reading_differs_only_by_row_factor():
    """The literal prefix-only softmax is the causal one rescaled per row on j < C."""
    hq, hkv, w, n, d = 2, 1, 4, 30, 8
    q = RNG.normal(size=(hq, w, d))
    k = RNG.normal(size=(hkv, n, d))
    Pa = O.window_attention(q, k, 0.5, normalise="causal_all")
    Pp = O.window_attention(q, k, 0.5, normalise="prefix")
    C = n - w
    ratio = Pp[:, :, :C] / Pa[:, :, :C]
    np.testing.assert_allclose(ratio, ratio[:, :, :1].repeat(C, axis=2), rtol=1e-12)
    np.testing.assert_allclose(ratio[:, :, 0], 1.0 / Pa[:, :, :C].sum(axis=2), rtol=1e-12)


# --------------------------------------------------------------------------
# Pooling, window reduction, GQA reduction
# --------------------------------------------------------------------------

@pytest.mark.parametrize("pool", [1, 3, 7])
def test_max_pool_matches_torch(pool):
    a = RNG.random(size=(5, 37))
    ref = torch.nn.functional.max_pool1d(torch.from_numpy(a)[None], pool, stride=1,
                                         padding=pool // 2)[0].numpy()
    np.testing.assert_array_equal(O.max_pool(a, pool), ref)


def test_window_reduce_equal_logits_closed_form():
    """q = 0: a[j] = (1/w) sum_t 1/(n-w+t+1), constant over j, so pooling leaves it unchanged."""
    hq, hkv, w, n, d = 4, 4, 8, 64, 4
    q = np.zeros((hq, w, d))
    k = RNG.normal(size=(hkv, n, d))
    s, _ = O.score_layer(q, k, k, w=w, pool=7)
    expect = np.mean([1.0 / (n - w + t + 1) for t in range(w)])
    np.testing.assert_allclose(s, expect, rtol=1e-13)
    assert s.shape == (hkv, n - w)


def test_pool_orders_differ_and_bracket():
    """max does not commute with the mean: pooling rows first can only be larger or equal."""
    hq, hkv, w, n, d = 2, 2, 6, 50, 8
    q = RNG.normal(size=(hq, w, d)) * 3
    k = RNG.normal(size=(hkv, n, d))
    P = O.window_attention(q, k, 0.4)
    a = O.window_reduce(P, n - w, 7, order="mean_then_pool")
    b = O.window_reduce(P, n - w, 7, order="pool_rows")
    assert np.all(b >= a - 1e-15)
    assert np.any(b > a + 1e-9)


def test_group_reduce_closed_form():
    p = np.array([[1.0, 4.0], [3.0, 0.0], [2.0, 2.0], [6.0, 1.0]])
    np.testing.assert_array_equal(O.group_reduce(p, 2, "mean"), [[2.0, 2.0], [4.0, 1.5]])
    np.testing.assert_array_equal(O.group_reduce(p, 2, "max"), [[3.0, 4.0], [6.0, 2.0]])
    np.testing.assert_array_equal(O.group_reduce(p, 4, "mean"), p)


def test_lava_and_critical_factors_closed_form():
    hkv, n, d, D, w = 2, 9, 4, 6, 3
    v = np.zeros((hkv, n, d))
    v[0, 4] = [1, -2, 0, 0]          # ||.||_1 = 3, the max of head 0
    v[0, 1] = [0.5, 0, 0, -0.5]
    v[1, 0] = [-1, -1, -1, -1]       # 4, the max of head 1
    np.testing.assert_array_equal(O.v_l1_max(v), [3.0, 4.0])
    # W^O with a single non-zero column e: ||(V W^O)_j||_1 = |V_j . col|.
    w_o = np.zeros((hkv, d, D))
    w_o[:, :, 2] = [1.0, 2.0, 3.0, 4.0]
    c = O.critical_row_norm(v, w_o, n - w)
    np.testing.assert_allclose(c[0, 4], abs(1 - 4), rtol=0)
    np.testing.assert_allclose(c[0, 1], abs(0.5 - 2.0), rtol=0)
    np.testing.assert_allclose(c[1, 0], 10.0, rtol=0)
    assert c.shape == (hkv, n - w)


def test_lava_score_is_vbar_times_group_max():
    hq, hkv, w, n, d = 4, 2, 4, 20, 8
    q = RNG.normal(size=(hq, w, d))
    k = RNG.normal(size=(hkv, n, d))
    v = RNG.normal(size=(hkv, n, d))
    s_ada_max, _ = O.score_layer(q, k, v, w=w, pool=7, mode="ada", group="max")
    s_lava, _ = O.score_layer(q, k, v, w=w, pool=7, mode="lava", group="max")
    np.testing.assert_allclose(s_lava, s_ada_max * O.v_l1_max(v)[:, None], rtol=1e-15)


# --------------------------------------------------------------------------
# Algorithm 1 and the Ada-KV theorems, by brute force on tiny inputs
# --------------------------------------------------------------------------

def _all_masks(h, C, B):
    for combo in itertools.combinations(range(h * C), B):
        T = np.zeros(h * C)
        T[list(combo)] = 1
        yield T.reshape(h, C)


@pytest.mark.parametrize("seed", range(6))
def test_theorem_3_3_global_topk_is_optimal(seed):
    """Global Top-B' retains the largest sum T*A over every mask with sum T = B'."""
    r = np.random.default_rng(seed)
    h, C = 3, 5
    A = r.dirichlet(np.ones(C) * 0.3, size=h)
    for Bp in (1, 4, 7, 11):
        f = O.global_topk_counts(A, Bp)
        assert f.sum() == Bp
        got = O.retained_mass(A, f)
        best = max(float((T * A).sum()) for T in _all_masks(h, C, Bp))
        assert got == pytest.approx(best, rel=0, abs=1e-14)
        # and so minimises eps of Theorem 3.1 over all allocations
        eps_got = O.eviction_bound(A, np.zeros_like(A), 1.0) - 2.0 * got
        eps_best = min(O.eviction_bound(A, T, 1.0) for T in _all_masks(h, C, Bp))
        assert eps_got == pytest.approx(eps_best, abs=1e-13)


@pytest.mark.parametrize("seed", range(4))
def test_theorem_3_2_per_head_topk_is_optimal(seed):
    r = np.random.default_rng(100 + seed)
    h, C = 2, 6
    A = r.dirichlet(np.ones(C), size=h)
    for Bg in [(1, 2), (3, 0), (2, 4)]:
        got = sum(A[g, O.topk_positions(A[g], Bg[g])].sum() for g in range(h))
        best = sum(max(A[g, list(cmb)].sum() for cmb in itertools.combinations(range(C), Bg[g]))
                   for g in range(h))
        assert got == pytest.approx(best, abs=1e-15)


@pytest.mark.parametrize("seed", range(8))
def test_theorem_3_1_loss_bound_holds(seed):
    """||y - yhat||_1 <= 2hC - 2C sum T*A with C the largest row L1 norm of V_i W_i^O."""
    r = np.random.default_rng(200 + seed)
    h, n, dh, D = 3, 12, 4, 10
    A = np.stack([O.row_softmax(r.normal(size=n) * 3) for _ in range(h)])
    V = r.normal(size=(h, n, dh))
    W = r.normal(size=(h, dh, D))
    VW = np.einsum("hnd,hde->hne", V, W)
    Cmax = float(np.abs(VW).sum(axis=2).max())
    y = sum(A[i] @ VW[i] for i in range(h))
    f = O.global_topk_counts(A, 10)
    T = np.zeros_like(A)
    for g in range(h):
        T[g, O.topk_positions(A[g], f[g])] = 1
    for g in range(h):     # every head keeps at least one element for yhat to exist
        if T[g].sum() == 0:
            T[g, np.argmax(A[g])] = 1
    yhat = O.masked_head_output(A, T, VW)
    assert np.abs(y - yhat).sum() <= O.eviction_bound(A, T, Cmax) + 1e-12


def test_flat_decode_equals_masked_softmax_output():
    """Decode over the compacted flat cache is the -inf-masked softmax of the Eviction Decision."""
    r = np.random.default_rng(7)
    hq, hkv, n, d, w, D = 4, 2, 30, 8, 5, 6
    k = r.normal(size=(hkv, n, d))
    v = r.normal(size=(hkv, n, d))
    s = r.random(size=(hkv, n - w))
    Bg = [7, 3]
    kept, cu, lens, Kf, Vf = O.compact_layer(k, v, s, Bg, w)
    q = r.normal(size=(hq, d))
    o, *_ = O.flat_decode(q, Kf, Vf, cu, lens, scale=0.35)
    G = hq // hkv
    for qh in range(hq):
        g = qh // G
        A = O.row_softmax(k[g] @ q[qh] * 0.35)[None]
        T = np.zeros((1, n))
        T[0, kept[g]] = 1
        Wid = np.eye(d)[None]
        yhat = O.masked_head_output(A, T, (v[g] @ Wid[0])[None])
        np.testing.assert_allclose(o[qh], yhat, rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------------------
# Safeguard blend (Ada-KV Algorithm 2, safeguard alpha)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(10))
def test_blend_invariants(seed):
    r = np.random.default_rng(300 + seed)
    H = int(r.integers(1, 9))
    C = int(r.integers(1, 40))
    s = r.random(size=(H, C)) ** 4
    Bp = int(r.integers(0, H * C + 1))
    f = O.global_topk_counts(s, Bp)
    for a, b in [(1, 5), (0, 1), (1, 1), (2, 7), (1, 2)]:
        Bg = O.safeguard_blend(f, Bp, a, b)
        assert Bg.sum() == Bp
        assert np.all(Bg >= (a * Bp) // (b * H))
        assert np.all(Bg <= C)
        if a == 0:
            np.testing.assert_array_equal(Bg, f)
        if a == b:  # alpha = 1: uniform SnapKV, remainder to the lowest heads
            q, rem = divmod(Bp, H)
            np.testing.assert_array_equal(Bg, [q + (1 if g < rem else 0) for g in range(H)])


def test_adaptive_mass_not_below_uniform():
    """Ada-KV Figure 1 analogue: blended budgets retain at least the uniform mass
    (concave per-head mass curves), up to one element per head of rounding."""
    r = np.random.default_rng(11)
    H, C = 8, 200
    temps = np.exp(r.uniform(np.log(0.5), np.log(16), size=H))
    s = np.stack([O.row_softmax(r.normal(size=C) * t) for t in temps])
    for Bp in (80, 400, 800):
        f = O.global_topk_counts(s, Bp)
        uni = O.safeguard_blend(f, Bp, 1, 1)
        ada = O.safeguard_blend(f, Bp, 1, 5)
        m_u = O.retained_mass(s, uni)
        m_a = O.retained_mass(s, ada)
        m_f = O.retained_mass(s, f)
        assert m_f >= m_a - 1e-12 >= m_u - H * s.max() - 1e-12
        assert m_a >= m_u - 1e-12


def test_head_budgets_validates_range():
    s = np.ones((2, 4))
    with pytest.raises(ValueError):
        O.head_budgets(s, B=2 * 3 - 1, w=3, a=1, b=5)
    with pytest.raises(ValueError):
        O.head_budgets(s, B=2 * 3 + 9, w=3, a=1, b=5)
    f, Bg = O.head_budgets(s, B=2 * 3 + 8, w=3, a=1, b=5)
    np.testing.assert_array_equal(Bg, [4, 4])


# --------------------------------------------------------------------------
# LAVa layer budgets and Theorem 1
# --------------------------------------------------------------------------

def test_layer_entropy_uniform_closed_form():
    hkv, C, n = 4, 50, 60
    s = np.full((hkv, C), 0.37)
    assert O.layer_entropy(s, n) == pytest.approx(math.log(hkv * C) / (hkv * n), rel=1e-14)
    z = np.zeros((hkv, C))
    z[1, 3] = 2.0       # a single non-zero score: zero entropy
    assert O.layer_entropy(z, n) == 0.0


def test_layer_budgets_sum_and_proportions():
    hkv, w, C = 2, 4, 100
    # equal entropies: uniform split, remainder to the lowest layers
    B = O.lava_layer_budgets([0.5, 0.5, 0.5], total=3 * 8 + 10, w=w, hkv=hkv, C=C)
    np.testing.assert_array_equal(B - w * hkv, [4, 3, 3])
    # proportional split 1:2:1 of R = 40
    B = O.lava_layer_budgets([0.25, 0.5, 0.25], total=3 * 8 + 40, w=w, hkv=hkv, C=C)
    np.testing.assert_array_equal(B - w * hkv, [10, 20, 10])
    # zero entropy layer gets nothing selectable
    B = O.lava_layer_budgets([0.0, 1.0], total=2 * 8 + 17, w=w, hkv=hkv, C=C)
    np.testing.assert_array_equal(B - w * hkv, [0, 17])
    # cap at Hkv*C: the overflow goes to the other layers
    B = O.lava_layer_budgets([0.9, 0.1, 0.0], total=3 * 8 + 250, w=w, hkv=hkv, C=C)
    np.testing.assert_array_equal(B - w * hkv, [200, 50, 0])
    r = np.random.default_rng(5)
    for _ in range(20):
        e = r.random(size=7)
        tot = 7 * 8 + int(r.integers(0, 7 * 2 * C))
        B = O.lava_layer_budgets(e, tot, w, hkv, C)
        assert B.sum() == tot
        assert np.all(B - w * hkv <= hkv * C) and np.all(B >= w * hkv)


@pytest.mark.parametrize("seed", range(6))
def test_lava_theorem_1_bound(seed):
    """||y - yhat||_1 <= 2 ||W_O^T||_1 sum_h sum_i A_h[i] Vbar_h (1 - T_h[i])."""
    r = np.random.default_rng(400 + seed)
    H, n, dh, D = 3, 14, 4, 9
    A = np.stack([O.row_softmax(r.normal(size=n) * 2) for _ in range(H)])
    V = r.normal(size=(H, n, dh)) * np.exp(0.5 * r.normal(size=(H, n, 1)))
    W = r.normal(size=(H * dh, D))
    vbar = O.v_l1_max(V)
    s = A * vbar[:, None]
    f = O.global_topk_counts(s, 12)
    T = np.zeros_like(A)
    for g in range(H):
        T[g, O.topk_positions(s[g], f[g])] = 1
        if T[g].sum() == 0:
            T[g, np.argmax(A[g])] = 1
    y = np.concatenate([A[h] @ V[h] for h in range(H)]) @ W
    yhat = np.concatenate([(A[h] * T[h] / (A[h] * T[h]).sum()) @ V[h] for h in range(H)]) @ W
    assert np.abs(y - yhat).sum() <= O.lava_bound(A, T, vbar, W) + 1e-12


# --------------------------------------------------------------------------
# Selection, compaction and decode
# --------------------------------------------------------------------------

def test_topk_positions_tie_order():
    s = np.array([0.2, 0.5, 0.2, 0.2, 0.5, 0.1])
    np.testing.assert_array_equal(O.topk_positions(s, 3), [0, 1, 4])
    np.testing.assert_array_equal(O.topk_positions(s, 4), [0, 1, 2, 4])
    np.testing.assert_array_equal(O.topk_positions(s, 0), [])


def test_critical_special_cases():
    r = np.random.default_rng(9)
    C = 40
    s = r.random(C) ** 3
    c = r.random(C) * 10
    for k in (0, 1, 7, 40):
        # alpha_c = 1: plain Top-k by s
        np.testing.assert_array_equal(O.critical_positions(s, c, k, 1, 1, 1e-6),
                                      O.topk_positions(s, k))
        # eps -> infinity: stage 2 ranks the rest by c alone
        got = O.critical_positions(s, c, k, 1, 2, 1e30)
        k1 = k // 2
        first = O.topk_positions(s, k1)
        rest = np.setdiff1d(np.arange(C), first)
        second = rest[np.argsort(-c[rest], kind="stable")[: k - k1]]
        np.testing.assert_array_equal(got, np.sort(np.concatenate([first, second])))


def test_compact_layout_and_window():
    r = np.random.default_rng(3)
    hkv, n, d, w = 3, 25, 4, 5
    k = r.normal(size=(hkv, n, d))
    v = r.normal(size=(hkv, n, d))
    s = r.random(size=(hkv, n - w))
    Bg = [0, 20, 6]
    kept, cu, lens, Kf, Vf = O.compact_layer(k, v, s, Bg, w, reserve=2)
    np.testing.assert_array_equal(lens, [5, 25, 11])
    np.testing.assert_array_equal(cu, [0, 7, 34, 47])
    for g in range(hkv):
        assert np.all(np.diff(kept[g]) > 0)
        np.testing.assert_array_equal(kept[g][-w:], np.arange(n - w, n))
        np.testing.assert_array_equal(Kf[cu[g]:cu[g] + lens[g]], k[g, kept[g]])
        assert np.all(Kf[cu[g] + lens[g]:cu[g + 1]] == 0)


def test_full_budget_decode_is_dense_attention_sdpa():
    """B = n*Hkv keeps everything: flat decode (with an append) equals SDPA over the full cache."""
    r = np.random.default_rng(21)
    hq, hkv, n, d, w = 8, 2, 33, 16, 4
    k = r.normal(size=(hkv, n, d))
    v = r.normal(size=(hkv, n, d))
    qw = r.normal(size=(hq, w, d))
    s, _ = O.score_layer(qw, k, v, w=w, pool=7)
    f, Bg = O.head_budgets(s, B=n * hkv, w=w, a=1, b=5)
    np.testing.assert_array_equal(Bg, [n - w] * hkv)
    kept, cu, lens, Kf, Vf = O.compact_layer(k, v, s, Bg, w, reserve=1)
    q = r.normal(size=(hq, d))
    kn = r.normal(size=(hkv, d))
    vn = r.normal(size=(hkv, d))
    scale = 1 / math.sqrt(d)
    o, _, _, lens2 = O.flat_decode(q, Kf, Vf, cu, lens, scale, kn, vn)
    np.testing.assert_array_equal(lens2, lens + 1)
    K2 = np.concatenate([k, kn[:, None]], axis=1)
    V2 = np.concatenate([v, vn[:, None]], axis=1)
    G = hq // hkv
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[:, None, None, :],
        torch.from_numpy(K2).repeat_interleave(G, 0)[:, None],
        torch.from_numpy(V2).repeat_interleave(G, 0)[:, None], scale=scale)[:, 0, 0].numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(O.dense_decode(q, K2, V2, scale), ref, rtol=1e-12, atol=1e-13)


def test_global_topk_tie_order():
    """Equal scores across heads go to the lower head first, then the lower position."""
    s = np.array([[0.5, 0.2], [0.2, 0.5]])
    np.testing.assert_array_equal(O.global_topk_counts(s, 3), [2, 1])
    s = np.array([[0.1, 0.3, 0.3], [0.3, 0.3, 0.0]])
    np.testing.assert_array_equal(O.global_topk_counts(s, 3), [2, 1])


def test_golden_ada_alg1_toy():
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "ada_alg1_toy.json")
    g = json.load(open(path))
    s = np.array(g["scores"])
    Bp = g["selectable_budget"]
    f = O.global_topk_counts(s, Bp)
    np.testing.assert_array_equal(f, g["counts"])
    for frac, expect in g["blend"].items():
        a, b = map(int, frac.split("/"))
        np.testing.assert_array_equal(O.safeguard_blend(f, Bp, a, b), expect)
    for key, expect in g["kept"].items():
        Bg = list(map(int, key.split(",")))
        for h in range(3):
            np.testing.assert_array_equal(O.topk_positions(s[h], Bg[h]), expect[h])
