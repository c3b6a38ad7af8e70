"""Full-size parity of the "next" paths, at the sizes bench.py times them.

- LAVa online prefill cascade on the 32-layer 128K workload: layer and head budgets at every
  stage bit-exact against the oracle's cascade fed the GPU's float32 scores, the final kept
  positions of every head bit-exact, and the gathered rows of sampled heads;
- GQA-exact CriticalKV and LaProx on the 32-layer 64K workload with one W_O block per query
  head: window terms and projected scores of sampled units within 1e-4 relative of the oracle
  (the norms on a seeded sample of rows), the two-stage selection and the model-wide LaProx
  budgets bit-exact when fed the GPU's own float32 scores.
"""
import math

import numpy as np
import pytest
import torch

import kv_cache_eviction_gb300 as kv
import oracle as O
from kv_cache_eviction_gb300 import workloads as W
from tests.kvpath import assert_scores_close, np64, run_allocate, run_score, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_eviction_gb300 import _build
    _build.build()
    kv.lib()


def test_cascade_fullsize_128k():
    wl = W.WORKLOADS["mistral7b_128k_lava"]
    L, hkv, n, w = wl.layers, wl.hkv, wl.n, wl.w
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    scores, _ = run_score(wl, shape, inp)
    total = wl.total_budget_value()
    reserve = 2
    cap = total + L * hkv * reserve
    flats = [{"kept": torch.full((cap,), -7, dtype=torch.int32, device="cuda"),
              "cu": torch.zeros(1, L, hkv + 1, dtype=torch.int64, device="cuda"),
              "lens": torch.zeros(1, L, hkv, dtype=torch.int32, device="cuda"),
              "kf": torch.zeros(cap, wl.d, dtype=torch.bfloat16, device="cuda"),
              "vf": torch.zeros(cap, wl.d, dtype=torch.bfloat16, device="cuda")}
             for _ in range(2)]
    caps = [torch.full((1, L), n * hkv, dtype=torch.int32, device="cuda") for _ in range(2)]
    budget = torch.tensor([total], dtype=torch.int64, device="cuda")
    w_a = workspace(kv.KV_OP_ALLOCATE, shape)
    w_r = torch.zeros(kv.kv_recompact_workspace_size(max(cap, hkv * n)), dtype=torch.uint8,
                      device="cuda")
    lbs, hbs = [], []
    for t in range(1, L + 1):
        sh_t = kv.KvShape.from_workload(wl, layers=t)
        lb = caps[t % 2]
        hb = torch.zeros(1, t, hkv, dtype=torch.int32, device="cuda")
        kv.kv_allocate_capped(sh_t, scores[:, :t], budget, caps[(t - 1) % 2], 0, 1, lb, hb, w_a)
        src, dst = flats[(t - 1) % 2], flats[t % 2]
        if t >= 2:
            kv.kv_recompact(kv.KvShape.from_workload(wl, layers=t - 1), scores[:, :t - 1],
                            hb[:, :t - 1].contiguous(), src["kept"], src["cu"][:, :t - 1],
                            src["lens"][:, :t - 1], src["kf"], src["vf"], reserve, None,
                            dst["kept"], dst["cu"], dst["lens"], dst["kf"], dst["vf"], w_r)
        row_base = dst["cu"][0, t - 2, hkv:hkv + 1] if t >= 2 else None
        kv.kv_recompact(kv.KvShape.from_workload(wl, layers=1), scores[:, t - 1:t],
                        hb[:, t - 1:t].contiguous(), None, None, None, inp["k"][:, t - 1:t],
                        inp["v"][:, t - 1:t], reserve, row_base, dst["kept"],
                        dst["cu"][:, t - 1:t], dst["lens"][:, t - 1:t], dst["kf"], dst["vf"], w_r)
        lbs.append(lb[0, :t].cpu().numpy().copy())
        hbs.append(hb[0].cpu().numpy().copy())
    assert kv.kv_check_device_status(w_a) == 0 and kv.kv_check_device_status(w_r) == 0
    final = flats[L % 2]
    S = [scores[0, l].double().cpu().numpy() for l in range(L)]
    ref = O.lava_cascade(S, total, w, n)
    for t in range(L):
        np.testing.assert_array_equal(lbs[t], ref[t]["layer_budget"], err_msg="stage %d" % (t + 1))
        np.testing.assert_array_equal(hbs[t], ref[t]["head_budget"], err_msg="stage %d" % (t + 1))
    kept = final["kept"].cpu().numpy()
    cu = final["cu"].cpu().numpy()[0]
    rng = np.random.default_rng(3)
    sampled = {(0, 0), (L - 1, hkv - 1)} | {(int(rng.integers(L)), int(rng.integers(hkv)))
                                             for _ in range(2)}
    for l in range(L):
        for g in range(hkv):
            k_ref = ref[-1]["kept"][l][g]
            r0 = int(cu[l, g])
            np.testing.assert_array_equal(kept[r0:r0 + len(k_ref)], k_ref)
            if (l, g) in sampled:
                kf = np64(final["kf"][r0:r0 + len(k_ref)])
                np.testing.assert_array_equal(kf, np64(inp["k"][0, l, g])[k_ref])


def test_per_query_head_scores_fullsize_64k():
    wl = W.WORKLOADS["llama8b_64k_criticalkv"]
    L, hkv, hq, n, w, D = wl.layers, wl.hkv, wl.hq, wl.n, wl.w, wl.model_dim
    G = hq // hkv
    C = n - w
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    g_ = torch.Generator(device="cuda").manual_seed(0x9A0)
    w_oq = (torch.randn(L, hq, wl.d, D, device="cuda", generator=g_) / math.sqrt(D)).to(
        torch.bfloat16)
    ws_s = workspace(kv.KV_OP_SCORE, shape)
    ws1 = torch.zeros(256, dtype=torch.uint8, device="cuda")
    scores, _ = run_score(wl, shape, inp, mode="ada")
    res = {}
    for name, tk, pk in (("crit", kv.KV_TERMS_MEAN_POOLED, kv.KV_PROJ_CRIT_GQA),
                         ("laprox", kv.KV_TERMS_L2, kv.KV_PROJ_LAPROX)):
        terms = torch.empty(1, L, hq, C, device="cuda")
        out = torch.empty(1, L, hkv, C, device="cuda")
        kv.kv_window_terms(shape, tk, inp["q_win"], inp["k"], terms, ws_s)
        kv.kv_proj_score(shape, pk, inp["v"], w_oq, D, terms, wl.crit_eps, out, ws1)
        assert kv.kv_check_device_status(ws_s) == 0 and kv.kv_check_device_status(ws1) == 0
        res[name] = (terms, out)
    pts = [(0, 0), (L - 1, hkv - 1), (13, 3), (22, 5)]
    for (l, g) in pts:
        q = np64(inp["q_win"][0, l, g * G:(g + 1) * G])
        k = np64(inp["k"][0, l, g:g + 1])
        v = np64(inp["v"][0, l, g:g + 1])
        for name, kind in (("crit", "mean_pool"), ("laprox", "l2")):
            terms, out = res[name]
            t_ref = O.window_head_terms(q, k, w, wl.pool, kind)
            t_gpu = terms[0, l, g * G:(g + 1) * G].double().cpu().numpy()
            assert_scores_close(t_gpu, t_ref, what="%s terms l%d g%d" % (name, l, g))
            rows = np.sort(np.random.default_rng(l * 31 + g).choice(C, size=128, replace=False))
            wq = np64(w_oq[l, g * G:(g + 1) * G])
            vr = v[:, rows]
            if name == "crit":
                ref = O.gqa_critical_kappa(t_gpu[:, rows], vr, wq, wl.crit_eps)[0]
            else:
                ref = O.laprox_score(t_gpu[:, rows], vr, wq)[0]
            got = out[0, l, g].double().cpu().numpy()[rows]
            assert_scores_close(got, ref, what="%s score l%d g%d" % (name, l, g))
    # selection fed the GPU's own scores: two-stage with kappa, and LaProx's model-wide TopK
    budgets = wl.budgets()
    _, hb = run_allocate(wl, shape, scores, budgets)
    cap = wl.flat_capacity_rows()
    kept = torch.empty(cap, dtype=torch.int32, device="cuda")
    cu = torch.empty(1, L, hkv + 1, dtype=torch.int64, device="cuda")
    lens = torch.empty(1, L, hkv, dtype=torch.int32, device="cuda")
    kf = torch.empty(cap, wl.d, dtype=torch.bfloat16, device="cuda")
    vf = torch.empty_like(kf)
    ws_c = workspace(kv.KV_OP_COMPACT, shape)
    kap = res["crit"][1]
    kv.kv_compact_kappa(shape, inp["k"], inp["v"], scores, kap, 1, 2, hb, wl.reserve, kept, cu,
                        lens, kf, vf, cap, ws_c)
    assert kv.kv_check_device_status(ws_c) == 0
    keptn, cun, hbn = kept.cpu().numpy(), cu.cpu().numpy()[0], hb.cpu().numpy()[0]
    s32, k32 = scores.cpu().numpy()[0], kap.cpu().numpy()[0]
    for (l, g) in pts:
        kg = int(hbn[l, g]) - w
        ref = O.critical_positions_kappa(s32[l, g].astype(np.float64),
                                         k32[l, g].astype(np.float64), kg, 1, 2)
        np.testing.assert_array_equal(keptn[cun[l, g]:cun[l, g] + kg], ref)
    p = res["laprox"][1]
    total = int(budgets.sum())
    lb = torch.empty(1, L, dtype=torch.int32, device="cuda")
    hb2 = torch.empty(1, L, hkv, dtype=torch.int32, device="cuda")
    ws_a = workspace(kv.KV_OP_ALLOCATE, shape)
    kv.kv_allocate(shape, p, torch.tensor([total], dtype=torch.int64, device="cuda"), 2, 0, 1,
                   lb, hb2, ws_a)
    assert kv.kv_check_device_status(ws_a) == 0
    p32 = p.cpu().numpy()[0]
    ref = O.laprox_head_budgets([p32[l].astype(np.float64) for l in range(L)], total, w)
    np.testing.assert_array_equal(hb2.cpu().numpy()[0], ref)
    np.testing.assert_array_equal(lb.cpu().numpy()[0], ref.sum(axis=1))
