"""Per-query-head scores on the GPU against the oracle: GQA-exact CriticalKV (one W_O block
per query head, group mean of (A_q + eps) * ||V W_O^q||_1, two-stage selection with that
key) and LaProx (||A_q[:, i]||_2 * ||(V W_O^q)_i||_2 summed over the group, one model-wide
TopK).

Bars: window terms and projected scores within 1e-4 relative of the oracle's fp64 values;
budgets and kept positions bit-exact when the selection is fed the oracle's scores (rounded
to float32); end to end, kept positions may differ only at near-ties.
"""
import math

import numpy as np
import pytest
import torch

import kv_cache_eviction_gb300 as kv
import oracle as O
from kv_cache_eviction_gb300 import workloads as W
from tests.kvpath import (assert_scores_close, capacity_rows, np64, oracle_kept_check,
                          run_allocate, workspace)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_eviction_gb300 import _build
    _build.build()
    kv.lib()


def setup(seed=5, L=2, n=1000, D=520):
    wl = W.Workload(name="gqa", batch=1, layers=L, hq=8, hkv=2, d=128, n=n, w=32, pool=7,
                    dtype="bf16", temp=(0.5, 16.0), mode="ada", head_budget_frac=0.3,
                    reserve=2, seed=seed)
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(seed + 1000)
    w_o = (torch.randn(L, wl.hq, wl.d, D, device="cuda", generator=g) / math.sqrt(D)).to(
        torch.bfloat16)
    return wl, shape, inp, w_o


def gpu_terms(wl, shape, inp, kind):
    C = wl.n - wl.w
    t = torch.full((1, wl.layers, wl.hq, C), float("nan"), device="cuda")
    ws = workspace(kv.KV_OP_SCORE, shape)
    kv.kv_window_terms(shape, kind, inp["q_win"], inp["k"], t, ws)
    assert kv.kv_check_device_status(ws) == 0
    return t


def gpu_proj(wl, shape, inp, w_o, terms, kind, eps):
    C = wl.n - wl.w
    out = torch.full((1, wl.layers, wl.hkv, C), float("nan"), device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    kv.kv_proj_score(shape, kind, inp["v"], w_o, w_o.shape[-1], terms, eps, out, ws)
    assert kv.kv_check_device_status(ws) == 0
    return out


@pytest.fixture(params=["tc", "simt"])
def score_path(request):
    """Window terms through the tcgen05 scoring kernel (its pass-2 epilogue writes every
    query head's window sums) and through the CUDA-core kernels."""
    import os
    old = os.environ.get("KVEVICT_SCORE_PATH")
    os.environ["KVEVICT_SCORE_PATH"] = request.param
    yield request.param
    if old is None:
        os.environ.pop("KVEVICT_SCORE_PATH", None)
    else:
        os.environ["KVEVICT_SCORE_PATH"] = old


@pytest.mark.parametrize("kind", [kv.KV_TERMS_MEAN_POOLED, kv.KV_TERMS_L2])
@pytest.mark.parametrize("n", [1000, 5000])
def test_window_terms_match_oracle(kind, n, score_path):
    wl, shape, inp, _ = setup(n=n, L=1 if n > 2000 else 2)
    t = gpu_terms(wl, shape, inp, kind).cpu().numpy()
    okind = "mean_pool" if kind == kv.KV_TERMS_MEAN_POOLED else "l2"
    for l in range(wl.layers):
        ref = O.window_head_terms(np64(inp["q_win"][0, l]), np64(inp["k"][0, l]), wl.w, wl.pool,
                                  okind)
        assert_scores_close(t[0, l].astype(np.float64), ref, what="terms %s l%d" % (okind, l))


@pytest.mark.parametrize("kind", [kv.KV_PROJ_CRIT_GQA, kv.KV_PROJ_LAPROX])
def test_proj_scores_match_oracle(kind):
    wl, shape, inp, w_o = setup()
    tk = kv.KV_TERMS_MEAN_POOLED if kind == kv.KV_PROJ_CRIT_GQA else kv.KV_TERMS_L2
    eps = 1e-3
    terms = gpu_terms(wl, shape, inp, tk)
    out = gpu_proj(wl, shape, inp, w_o, terms, kind, eps).cpu().numpy()
    tt = terms.double().cpu().numpy()
    for l in range(wl.layers):
        v = np64(inp["v"][0, l])
        wq = np64(w_o[l])
        if kind == kv.KV_PROJ_CRIT_GQA:
            ref = O.gqa_critical_kappa(tt[0, l], v, wq, eps)
        else:
            ref = O.laprox_score(tt[0, l], v, wq)
        assert_scores_close(out[0, l].astype(np.float64), ref, what="proj %d l%d" % (kind, l))


def _flat_out(wl, cap):
    return {"kept": torch.full((cap,), -7, dtype=torch.int32, device="cuda"),
            "cu": torch.empty(1, wl.layers, wl.hkv + 1, dtype=torch.int64, device="cuda"),
            "lens": torch.empty(1, wl.layers, wl.hkv, dtype=torch.int32, device="cuda"),
            "kf": torch.zeros(cap, wl.d, dtype=torch.bfloat16, device="cuda"),
            "vf": torch.zeros(cap, wl.d, dtype=torch.bfloat16, device="cuda")}


def test_gqa_criticalkv_two_stage_fed_and_end_to_end():
    wl, shape, inp, w_o = setup(seed=9)
    eps = 1e-3
    C = wl.n - wl.w
    # GPU scores: the Ada score (stage 1, allocation) and the GQA-exact kappa (stage 2)
    ws_s = workspace(kv.KV_OP_SCORE, shape)
    scores = torch.empty(1, wl.layers, wl.hkv, C, device="cuda")
    kv.kv_score(shape, kv.KV_SCORE_ADA, kv.KV_GROUP_MEAN, inp["q_win"], inp["k"], None, None, 0,
                scores, None, ws_s)
    terms = gpu_terms(wl, shape, inp, kv.KV_TERMS_MEAN_POOLED)
    kap = gpu_proj(wl, shape, inp, w_o, terms, kv.KV_PROJ_CRIT_GQA, eps)
    # oracle
    s_ref = np.zeros((wl.layers, wl.hkv, C))
    k_ref = np.zeros((wl.layers, wl.hkv, C))
    for l in range(wl.layers):
        q, k, v = np64(inp["q_win"][0, l]), np64(inp["k"][0, l]), np64(inp["v"][0, l])
        s_ref[l], _ = O.score_layer(q, k, v, w=wl.w, pool=wl.pool)
        tq = O.window_head_terms(q, k, wl.w, wl.pool, "mean_pool")
        k_ref[l] = O.gqa_critical_kappa(tq, v, np64(w_o[l]), eps)
    budgets = wl.budgets()
    cap = capacity_rows(wl, 1, wl.layers, budgets)
    ws_c = workspace(kv.KV_OP_COMPACT, shape)
    for fed in (True, False):
        s_in = torch.from_numpy(s_ref.astype(np.float32))[None].cuda() if fed else scores
        k_in = torch.from_numpy(k_ref.astype(np.float32))[None].cuda() if fed else kap
        _, hb = run_allocate(wl, shape, s_in, budgets)
        f = _flat_out(wl, cap)
        kv.kv_compact_kappa(shape, inp["k"], inp["v"], s_in, k_in, 1, 2, hb, wl.reserve, f["kept"],
                            f["cu"], f["lens"], f["kf"], f["vf"], cap, ws_c)
        assert kv.kv_check_device_status(ws_c) == 0
        kept, cu, hbn = f["kept"].cpu().numpy(), f["cu"].cpu().numpy(), hb.cpu().numpy()
        s32, k32 = s_in.cpu().numpy(), k_in.cpu().numpy()
        for l in range(wl.layers):
            for g in range(wl.hkv):
                kg = int(hbn[0, l, g]) - wl.w
                got = kept[cu[0, l, g]:cu[0, l, g] + kg]
                if fed:
                    ref = O.critical_positions_kappa(s32[0, l, g].astype(np.float64),
                                                     k32[0, l, g].astype(np.float64), kg, 1, 2)
                    np.testing.assert_array_equal(got, ref)
                else:
                    # end to end: stage 1 from the GPU's own scores, then kappa near-ties only
                    k1 = kg // 2
                    order = np.lexsort((got, -s32[0, l, g][got].astype(np.float64)))
                    st1 = np.sort(got[order[:k1]])
                    oracle_kept_check(s_ref[l, g], st1, k1)
                    rest = np.setdiff1d(np.arange(C), st1)
                    st2 = np.setdiff1d(got, st1)
                    oracle_kept_check(np.where(np.isin(np.arange(C), rest), k_ref[l, g], -1.0),
                                      st2, kg - k1)
                # the window follows
                np.testing.assert_array_equal(kept[cu[0, l, g] + kg:cu[0, l, g] + kg + wl.w],
                                              np.arange(C, wl.n))


def test_laprox_model_wide_selection_fed_and_end_to_end():
    wl, shape, inp, w_o = setup(seed=13, L=3)
    C = wl.n - wl.w
    terms = gpu_terms(wl, shape, inp, kv.KV_TERMS_L2)
    p_gpu = gpu_proj(wl, shape, inp, w_o, terms, kv.KV_PROJ_LAPROX, 0.0)
    p_ref = []
    for l in range(wl.layers):
        q, k, v = np64(inp["q_win"][0, l]), np64(inp["k"][0, l]), np64(inp["v"][0, l])
        p_ref.append(O.laprox_score(O.window_head_terms(q, k, wl.w, wl.pool, "l2"), v,
                                    np64(w_o[l])))
    total = wl.layers * wl.hkv * (wl.w + 150)
    budget = torch.tensor([total], dtype=torch.int64, device="cuda")
    cap = total + wl.layers * wl.hkv * wl.reserve
    ws_a = workspace(kv.KV_OP_ALLOCATE, shape)
    ws_c = workspace(kv.KV_OP_COMPACT, shape)
    for fed in (True, False):
        p_in = (torch.from_numpy(np.stack(p_ref).astype(np.float32))[None].cuda() if fed
                else p_gpu)
        lb = torch.empty(1, wl.layers, dtype=torch.int32, device="cuda")
        hb = torch.empty(1, wl.layers, wl.hkv, dtype=torch.int32, device="cuda")
        kv.kv_allocate(shape, p_in, budget, 2, 0, 1, lb, hb, ws_a)
        assert kv.kv_check_device_status(ws_a) == 0
        hbn = hb.cpu().numpy()[0]
        np.testing.assert_array_equal(lb.cpu().numpy()[0], hbn.sum(axis=1))
        assert hbn.sum() == total
        p32 = p_in.cpu().numpy()[0]
        if fed:
            ref = O.laprox_head_budgets([p32[l].astype(np.float64) for l in range(wl.layers)],
                                        total, wl.w)
            np.testing.assert_array_equal(hbn, ref)
        f = _flat_out(wl, cap)
        kv.kv_compact(shape, inp["k"], inp["v"], p_in, None, 1, 2, 0.0, hb, wl.reserve,
                      f["kept"], f["cu"], f["lens"], f["kf"], f["vf"], cap, ws_c)
        assert kv.kv_check_device_status(ws_c) == 0
        kept, cu = f["kept"].cpu().numpy(), f["cu"].cpu().numpy()
        for l in range(wl.layers):
            for g in range(wl.hkv):
                kg = int(hbn[l, g]) - wl.w
                got = kept[cu[0, l, g]:cu[0, l, g] + kg]
                if fed:
                    np.testing.assert_array_equal(got, O.topk_positions(
                        p32[l, g].astype(np.float64), kg))
                else:
                    oracle_kept_check(p_ref[l][g], got, kg)
