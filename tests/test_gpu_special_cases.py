"""Special cases of the method that fix the GPU path's results without the oracle.

Each reduces the path to a simpler result stated independently of it:
- alpha = 1 (all weight on the uniform share) gives SnapKV's uniform per-head budgets: B'/Hkv
  each, the remainder one by one to the lowest heads (Ada-KV Algorithm 2, safeguard);
- alpha = 0 keeps, per layer, exactly the layer-wide top-B' candidates in the total order
  (score desc, head asc, position asc): the per-head top-f_g sets of Ada-KV Algorithm 1
  together are the layer's top-B';
- CriticalKV with alpha_c = 1 (its first stage takes the whole budget) keeps what Ada-KV keeps;
- LAVa with max_k ||V[k]||_1 equal across a layer's heads ranks like Ada-KV: with that factor
  a power of two its scores are exactly Ada-KV's times it, and every selection is the same.
"""
import numpy as np
import pytest
import torch

import kv_cache_eviction_gb300 as kv
from kv_cache_eviction_gb300 import workloads as W
from tests.kvpath import capacity_rows, run_allocate, run_compact, run_score

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_eviction_gb300 import _build
    _build.build()
    kv.lib()


def base_workload(**kw):
    # two 16K layers, 40 % of n per head plus 5 rows so that B' / Hkv leaves a remainder
    wl = W.WORKLOADS["llama8b_16k_layer"].with_(layers=2, head_budget_frac=None,
                                                layer_budget=8 * 6553 + 5)
    return wl.with_(**kw)


def test_alpha_one_gives_uniform_budgets():
    wl = base_workload(alpha=(1, 1))
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    scores, _ = run_score(wl, shape, inp)
    _, hb = run_allocate(wl, shape, scores, wl.budgets())
    Bp = wl.layer_budget_value() - wl.w * wl.hkv
    expect = np.array([Bp // wl.hkv + (1 if g < Bp % wl.hkv else 0) for g in range(wl.hkv)])
    assert Bp % wl.hkv != 0
    got = hb.cpu().numpy() - wl.w
    for b in range(wl.batch):
        for l in range(wl.layers):
            np.testing.assert_array_equal(got[b, l], expect)


def test_alpha_zero_keeps_the_layer_wide_top():
    wl = base_workload(alpha=(0, 1))
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    scores, _ = run_score(wl, shape, inp)
    _, hb = run_allocate(wl, shape, scores, wl.budgets())
    cap = capacity_rows(wl, wl.batch, wl.layers, wl.budgets())
    flat = run_compact(wl, shape, inp, scores, None, hb, cap)
    s = scores.cpu().numpy()
    kept, cu, hbn = flat["kept"].cpu().numpy(), flat["cu"].cpu().numpy(), hb.cpu().numpy()
    Bp = wl.layer_budget_value() - wl.w * wl.hkv
    C = wl.n - wl.w
    g_idx, j_idx = np.meshgrid(np.arange(wl.hkv), np.arange(C), indexing="ij")
    for b in range(wl.batch):
        for l in range(wl.layers):
            sl = s[b, l]
            order = np.lexsort((j_idx.ravel(), g_idx.ravel(), -sl.ravel()))
            top = order[:Bp]
            expect = set(zip(g_idx.ravel()[top].tolist(), j_idx.ravel()[top].tolist()))
            got = set()
            for g in range(wl.hkv):
                k = int(hbn[b, l, g]) - wl.w
                base = int(cu[b, l, g])
                got.update((g, int(j)) for j in kept[base:base + k])
                # the window rows follow the candidates
                np.testing.assert_array_equal(kept[base + k:base + k + wl.w],
                                              np.arange(C, wl.n))
            assert got == expect


def test_criticalkv_full_first_stage_is_ada():
    wl = W.WORKLOADS["llama8b_64k_criticalkv"].with_(layers=2, n=8192, model_dim=1024,
                                                     crit_alpha=(1, 1))
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    scores, crit = run_score(wl, shape, inp)
    _, hb = run_allocate(wl, shape, scores, wl.budgets())
    cap = capacity_rows(wl, wl.batch, wl.layers, wl.budgets())
    with_crit = run_compact(wl, shape, inp, scores, crit, hb, cap)
    ada = run_compact(wl, shape, inp, scores, None, hb, cap)
    for k in ("kept", "cu", "lens", "kf", "vf"):
        assert torch.equal(with_crit[k], ada[k]), k


def test_lava_with_equal_vbar_ranks_like_ada():
    wl = base_workload(alpha=(0, 1))
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    # every head's largest ||V[k]||_1 is row 0, all ones: 128 in every head, a power of two
    v = inp["v"]
    v.mul_(0.01)
    v[:, :, :, 0, :] = 1.0
    ada, _ = run_score(wl, shape, inp, mode="ada", group="mean")
    lava, _ = run_score(wl, shape, inp, mode="lava", group="mean")
    assert torch.equal(lava, ada * float(wl.d))
    cap = capacity_rows(wl, wl.batch, wl.layers, wl.budgets())
    outs = []
    for sc in (ada, lava):
        lb, hb = run_allocate(wl, shape, sc, wl.budgets())
        outs.append((hb, run_compact(wl, shape, inp, sc, None, hb, cap)))
    assert torch.equal(outs[0][0], outs[1][0])
    for k in ("kept", "cu", "lens"):
        assert torch.equal(outs[0][1][k], outs[1][1][k]), k
