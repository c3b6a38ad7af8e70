"""Pins of the oracle's per-query-head scores (GQA-exact CriticalKV, LaProx) against what the
pages and the mathematics fix, independently of the functions under test:

- the per-head window mean, pooled, averaged over a group is Ada-KV's score (score_layer,
  pinned in test_oracle_pins);
- ||A[:, j]||_2 at q = 0 is the closed form sqrt(sum_t (C + t + 1)^-2), and lies between
  ||A[:, j]||_1 / sqrt(w) and ||A[:, j]||_1;
- ||(V W^O_q)_j||_1 with one block per group is critical_row_norm; ||.||_2 through a W^O with
  orthonormal rows is ||V_j||_2;
- with one W^O block shared by a group, the GQA-exact stage-2 key is (s + eps) * c, and its
  two-stage selection is critical_positions';
- LaProx's score for one head is the Frobenius norm of the entry's rank-one contribution
  A[:, i] (x) H[i, :], formed explicitly; its model-wide TopK keeps the subset of largest
  total score (brute force over every subset on tiny inputs).
"""
import itertools
import math

import numpy as np
import pytest

import oracle as O


def make(seed, hq=8, hkv=2, n=40, w=6, d=16, D=24):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((hq, w, d)) * 2
    k = rng.standard_normal((hkv, n, d))
    v = rng.standard_normal((hkv, n, d))
    w_o = rng.standard_normal((hq, d, D)) / math.sqrt(D)
    return q, k, v, w_o


@pytest.mark.parametrize("seed", range(3))
def test_mean_pool_terms_group_mean_is_the_ada_score(seed):
    q, k, v, _ = make(seed)
    t = O.window_head_terms(q, k, w=6, pool=5, kind="mean_pool")
    s, _ = O.score_layer(q, k, v, w=6, pool=5)
    G = q.shape[0] // k.shape[0]
    np.testing.assert_allclose(t.reshape(k.shape[0], G, -1).mean(axis=1), s, rtol=1e-12)


def test_l2_terms_closed_form_at_zero_query():
    hq, hkv, n, w, d = 4, 2, 30, 5, 8
    q = np.zeros((hq, w, d))
    k = np.random.default_rng(1).standard_normal((hkv, n, d))
    t = O.window_head_terms(q, k, w=w, pool=1, kind="l2")
    C = n - w
    ref = math.sqrt(sum((1.0 / (C + tt + 1)) ** 2 for tt in range(w)))
    np.testing.assert_allclose(t, np.full((hq, C), ref), rtol=1e-12)


def test_l2_terms_between_norm_bounds():
    q, k, v, _ = make(4)
    w = q.shape[1]
    l2 = O.window_head_terms(q, k, w=w, pool=1, kind="l2")
    l1 = O.window_head_terms(q, k, w=w, pool=1, kind="mean_pool") * w   # pool 1: no pooling
    assert np.all(l2 <= l1 * (1 + 1e-12)) and np.all(l2 >= l1 / math.sqrt(w) * (1 - 1e-12))


def test_proj_norm_l1_with_shared_blocks_is_critical_row_norm():
    q, k, v, w_o = make(5)
    hq, hkv = q.shape[0], k.shape[0]
    G = hq // hkv
    shared = np.repeat(w_o[::G], G, axis=0)          # block of query head g*G for its group
    C = k.shape[1] - q.shape[1]
    got = O.head_proj_norm(v, shared, C, 1)
    ref = O.critical_row_norm(v, w_o[::G], C)
    np.testing.assert_allclose(got.reshape(hkv, G, C), np.repeat(ref[:, None], G, axis=1),
                               rtol=1e-12)


def test_proj_norm_l2_through_orthonormal_rows_is_the_row_norm():
    rng = np.random.default_rng(6)
    hkv, hq, n, d, D = 2, 4, 20, 8, 16
    v = rng.standard_normal((hkv, n, d))
    blocks = []
    for _ in range(hq):
        Q, _ = np.linalg.qr(rng.standard_normal((D, D)))
        blocks.append(Q[:d])                          # d orthonormal rows of length D
    w_o = np.stack(blocks)
    got = O.head_proj_norm(v, w_o, n, 2)
    G = hq // hkv
    for qh in range(hq):
        np.testing.assert_allclose(got[qh], np.sqrt((v[qh // G] ** 2).sum(axis=1)), rtol=1e-10)


@pytest.mark.parametrize("seed", range(3))
def test_gqa_kappa_with_shared_blocks_is_the_per_kv_head_form(seed):
    q, k, v, w_o = make(seed + 10)
    hq, hkv = q.shape[0], k.shape[0]
    G = hq // hkv
    shared = np.repeat(w_o[::G], G, axis=0)
    w, pool, eps = q.shape[1], 5, 1e-3
    C = k.shape[1] - w
    terms = O.window_head_terms(q, k, w=w, pool=pool, kind="mean_pool")
    kap = O.gqa_critical_kappa(terms, v, shared, eps)
    s, c = O.score_layer(q, k, v, w=w, pool=pool, mode="critical", w_o=w_o[::G])
    np.testing.assert_allclose(kap, (s + eps) * c, rtol=1e-12)
    for g in range(hkv):
        for kk in (0, 7, 20, C):
            np.testing.assert_array_equal(
                O.critical_positions_kappa(s[g], kap[g], kk, 1, 2),
                O.critical_positions(s[g], c[g], kk, 1, 2, eps))


def test_kappa_selection_alpha_one_is_plain_topk():
    rng = np.random.default_rng(3)
    s = rng.random(50)
    kap = rng.random(50)
    for kk in (0, 5, 50):
        np.testing.assert_array_equal(O.critical_positions_kappa(s, kap, kk, 1, 1),
                                      O.topk_positions(s, kk))


def test_laprox_mha_score_is_the_frobenius_norm_of_the_contribution():
    q, k, v, w_o = make(20, hq=2, hkv=2)
    w = q.shape[1]
    C = k.shape[1] - w
    terms = O.window_head_terms(q, k, w=w, pool=1, kind="l2")
    p = O.laprox_score(terms, v, w_o)
    P = O.window_attention(q, k, 1.0 / math.sqrt(q.shape[2]))
    for h in range(2):
        H = v[h] @ w_o[h]
        for i in (0, 3, C - 1):
            contrib = np.outer(P[h, :, i], H[i])          # the entry's share of the outputs
            np.testing.assert_allclose(p[h, i], math.sqrt((contrib ** 2).sum()), rtol=1e-10)


def test_laprox_topk_keeps_the_largest_total_by_brute_force():
    rng = np.random.default_rng(8)
    L, hkv, C, w = 2, 2, 3, 1
    for _ in range(20):
        P = [np.round(rng.random((hkv, C)), 1) for _ in range(L)]   # rounding makes ties
        for Bp in range(0, L * hkv * C + 1):
            hb = O.laprox_head_budgets(P, Bp + L * w * hkv, w) - w
            flat = np.concatenate(P).reshape(-1)
            best = max(sum(flat[list(c)]) for c in itertools.combinations(range(flat.size), Bp))
            # the counts of the first Bp entries by (score desc, index asc) reach the best sum
            got = sum(np.sort(np.concatenate(P)[i])[::-1][:hb.reshape(-1)[i]].sum()
                      for i in range(L * hkv))
            assert abs(got - best) < 1e-9
            assert hb.sum() == Bp
