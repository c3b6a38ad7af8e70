"""The per-head selection's two kernels on the same scores.

kv_compact selects with the span of each CTA staged in shared memory (candidate lists
bounded by the largest key of each group of 4) when the span fits, and otherwise with the
kernel that reads the scores from global memory on every pass; KVEVICT_SELECT_PATH=global
forces the latter.  Kept indices, offsets and lengths must be identical.  The shapes cover
long spans with short lists, lists that overflow (large budgets, all-tied scores),
CriticalKV's two stages and ragged tiny spans; the oracle's top-k checks the 128K heads.
"""
import os

import numpy as np
import pytest
import torch

import kv_cache_eviction_gb300 as kv
import oracle as O
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


def compact_path(path, wl, shape, inp, scores, crit, hb, cap):
    old = os.environ.get("KVEVICT_SELECT_PATH")
    if path is None:
        os.environ.pop("KVEVICT_SELECT_PATH", None)
    else:
        os.environ["KVEVICT_SELECT_PATH"] = path
    try:
        flat = run_compact(wl, shape, inp, scores, crit, hb, cap)
        torch.cuda.synchronize()
        return {k: flat[k].cpu().numpy() for k in ("kept", "cu", "lens")}
    finally:
        if old is None:
            os.environ.pop("KVEVICT_SELECT_PATH", None)
        else:
            os.environ["KVEVICT_SELECT_PATH"] = old


def both_paths(wl, shape, inp, scores, crit, hb, cap):
    a = compact_path(None, wl, shape, inp, scores, crit, hb, cap)
    b = compact_path("global", wl, shape, inp, scores, crit, hb, cap)
    for k in ("kept", "cu", "lens"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    return a


def check_topk(out, s32, hb, w):
    """Non-CriticalKV selection: each head's kept candidates are the oracle's top-B_g of the
    same float32 scores (score desc, position asc), in ascending order."""
    B, L, H, C = s32.shape
    for b in range(B):
        for l in range(L):
            for g in range(H):
                bg = int(hb[b, l, g]) - w
                base = int(out["cu"][b, l, g])
                ref = O.topk_positions(s32[b, l, g].astype(np.float64), bg)
                np.testing.assert_array_equal(out["kept"][base:base + bg], ref,
                                              err_msg="head %d/%d/%d" % (b, l, g))


@pytest.fixture(scope="module")
def lava_128k():
    wl = W.WORKLOADS["mistral7b_128k_lava"].with_(layers=1)
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    scores, _ = run_score(wl, shape, inp)
    return wl, shape, inp, scores


def test_long_spans_short_lists(lava_128k):
    wl, shape, inp, scores = lava_128k
    budgets = wl.budgets()
    _, hb = run_allocate(wl, shape, scores, budgets)
    cap = capacity_rows(wl, wl.batch, wl.layers, budgets)
    out = both_paths(wl, shape, inp, scores, None, hb, cap)
    check_topk(out, scores.cpu().numpy(), hb.cpu().numpy(), wl.w)


@pytest.mark.parametrize("frac", [0.05, 0.6])
def test_large_budgets_overflow_the_lists(lava_128k, frac):
    wl, shape, inp, scores = lava_128k
    C = wl.n - wl.w
    rng = np.random.default_rng(int(frac * 100))
    bg = (frac * C * rng.uniform(0.5, 1.5, size=(1, 1, wl.hkv))).astype(np.int64)
    bg = np.clip(bg, 0, C)
    hb = torch.from_numpy((bg + wl.w).astype(np.int32)).cuda()
    cap = int(hb.sum()) + wl.hkv * wl.reserve
    out = both_paths(wl, shape, inp, scores, None, hb, cap)
    check_topk(out, scores.cpu().numpy(), hb.cpu().numpy(), wl.w)


def test_all_tied_scores_keep_the_lowest_positions(lava_128k):
    wl, shape, inp, scores = lava_128k
    C = wl.n - wl.w
    tied = torch.full_like(scores, 0.375)
    bg = np.array([0, 1, 31, 32, 33, 1000, C // 2, C], dtype=np.int64)[: wl.hkv]
    hb = torch.from_numpy((bg + wl.w).astype(np.int32).reshape(1, 1, -1)).cuda()
    cap = int(hb.sum()) + wl.hkv * wl.reserve
    out = both_paths(wl, shape, inp, tied, None, hb, cap)
    for g in range(wl.hkv):
        base = int(out["cu"][0, 0, g])
        np.testing.assert_array_equal(out["kept"][base:base + bg[g]], np.arange(bg[g]))


def test_criticalkv_two_stages():
    wl = W.WORKLOADS["llama8b_64k_criticalkv"].with_(n=8192, layers=2, model_dim=1024)
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    scores, crit = run_score(wl, shape, inp)
    budgets = wl.budgets()
    _, hb = run_allocate(wl, shape, scores, budgets)
    cap = capacity_rows(wl, wl.batch, wl.layers, budgets)
    both_paths(wl, shape, inp, scores, crit, hb, cap)


def test_ragged_tiny_spans():
    wl = W.Workload(name="tiny_spans", batch=2, layers=3, hq=8, hkv=4, d=64, n=77 + 13, w=13,
                    pool=5, dtype="bf16", temp=(0.5, 16.0), head_budget_tokens=40, reserve=2,
                    seed=321)
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    scores, _ = run_score(wl, shape, inp)
    budgets = wl.budgets()
    _, hb = run_allocate(wl, shape, scores, budgets)
    cap = capacity_rows(wl, wl.batch, wl.layers, budgets)
    out = both_paths(wl, shape, inp, scores, None, hb, cap)
    check_topk(out, scores.cpu().numpy(), hb.cpu().numpy(), wl.w)
