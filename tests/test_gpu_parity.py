"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, on seeded inputs.

Bars: scores within 1e-4 relative (+1e-12 absolute); budgets, kept indices, offsets and
the gathered rows bit-exact when the selection kernels are fed the oracle's scores
(rounded to float32, the kernels' input type); end to end, a kept index may differ only
at a near-tie (oracle score gap <= 1e-5 of the head's threshold); decode outputs within
1e-2 max-abs for bf16 (float32 accumulation on the GPU) and 1e-4 for float32.  The bf16 bar
applies to the accumulated value: where |o| < 4 it is asserted as a plain 1e-2, and where
|o| >= 4 the output's own bf16 storage rounding (half an ulp, at most 2^-8 |o|) is added,
since no bf16 value there need lie within a plain 1e-2 (`tests.kvpath.assert_decode_close`).
"""
import math

import numpy as np
import pytest
import torch

import kv_cache_eviction_gb300 as kv
import oracle as O
from kv_cache_eviction_gb300 import workloads as W
from tests.kvpath import (assert_decode_close, assert_scores_close, capacity_rows, np64,
                          oracle_crit_kept_check, oracle_kept_check, run_allocate, run_compact,
                          run_decode, run_score)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_eviction_gb300 import _build
    _build.build()
    kv.lib()


def oracle_scores(wl, q, k, v, w_o=None, mode=None, group=None):
    """Oracle scores of one (sequence, layer), one KV head at a time (heads are independent)."""
    mode = wl.mode if mode is None else mode
    group = wl.group if group is None else group
    G = wl.hq // wl.hkv
    S, Cn = [], []
    for g in range(wl.hkv):
        s, c = O.score_layer(q[g * G:(g + 1) * G], k[g:g + 1], v[g:g + 1], w=wl.w, pool=wl.pool,
                             mode=mode, group=group,
                             w_o=None if w_o is None else w_o[g:g + 1])
        S.append(s[0])
        if c is not None:
            Cn.append(c[0])
    return np.stack(S), (np.stack(Cn) if Cn else None)


def unit_np(inp, b, l, wl):
    q = np64(inp["q_win"][b, l])
    k = np64(inp["k"][b, l])
    v = np64(inp["v"][b, l])
    w_o = np64(inp["w_o"][l]) if inp.get("w_o") is not None else None
    return q, k, v, w_o


def check_fed_oracle_scores(wl, shape, inp, s32_all, c32_all, budgets, alpha=None):
    """Integer outputs are bit-exact when the selection kernels get the oracle's scores."""
    dev = "cuda"
    B, L = shape.batch, shape.layers
    s_t = torch.from_numpy(s32_all).to(dev)
    c_t = torch.from_numpy(c32_all).to(dev) if c32_all is not None else None
    a, b_ = wl.alpha if alpha is None else alpha
    lb, hb = run_allocate(wl, shape, s_t, budgets, alpha=(a, b_))
    lb, hb = lb.cpu().numpy(), hb.cpu().numpy()
    cap = capacity_rows(wl, B, L, budgets)
    flat = run_compact(wl, shape, inp, s_t, c_t, torch.from_numpy(hb).to(dev), cap)
    kept = flat["kept"].cpu().numpy()
    cu = flat["cu"].cpu().numpy()
    lens = flat["lens"].cpu().numpy()
    kf = np64(flat["kf"])
    vf = np64(flat["vf"])
    oracle_flat = {}
    running = 0
    for bb in range(B):
        s64 = s32_all[bb].astype(np.float64)
        if wl.budget_kind == "total":
            e = [O.layer_entropy(s64[l], wl.n) for l in range(L)]
            lb_ref = O.lava_layer_budgets(e, int(budgets[bb]), wl.w, wl.hkv, wl.n - wl.w)
            np.testing.assert_array_equal(lb[bb], lb_ref)
        else:
            lb_ref = budgets[bb].numpy()
            np.testing.assert_array_equal(lb[bb], lb_ref)
        for l in range(L):
            f, Bg = O.head_budgets(s64[l], int(lb_ref[l]), wl.w, a, b_)
            np.testing.assert_array_equal(hb[bb, l], Bg + wl.w)
            q, k, v, _ = unit_np(inp, bb, l, wl)
            crit = None
            c64 = None
            if c32_all is not None:
                crit = (wl.crit_alpha[0], wl.crit_alpha[1], wl.crit_eps)
                c64 = c32_all[bb, l].astype(np.float64)
            kept_r, cu_r, lens_r, Kf, Vf = O.compact_layer(
                k, v, s64[l], Bg, wl.w, reserve=wl.reserve, c=c64, crit=crit,
                kappa_dtype=np.float32)
            oracle_flat[(bb, l)] = (cu_r, lens_r, Kf, Vf)
            np.testing.assert_array_equal(cu[bb, l] - cu[bb, l, 0], cu_r)
            assert cu[bb, l, 0] == running
            running = cu[bb, l, -1]
            np.testing.assert_array_equal(lens[bb, l], lens_r)
            for g in range(wl.hkv):
                base = cu[bb, l, g]
                np.testing.assert_array_equal(kept[base:base + lens_r[g]], kept_r[g])
                assert np.all(kept[base + lens_r[g]:cu[bb, l, g + 1]] == -1)
            base = cu[bb, l, 0]
            np.testing.assert_array_equal(kf[base:base + len(Kf)][_filled(cu_r, lens_r)],
                                          Kf[_filled(cu_r, lens_r)])
            np.testing.assert_array_equal(vf[base:base + len(Vf)][_filled(cu_r, lens_r)],
                                          Vf[_filled(cu_r, lens_r)])
    return flat, oracle_flat


def _filled(cu, lens):
    idx = []
    for g in range(len(lens)):
        idx.extend(range(cu[g], cu[g] + lens[g]))
    return np.array(idx, dtype=np.int64)


def decode_and_check(wl, shape, flat, oracle_flat, steps, tau, atol):
    """Decode `steps` steps with appends on the GPU; the oracle replays them on its own flat
    cache (which the fed-scores check proved identical to the GPU's)."""
    B, L = shape.batch, shape.layers
    scale = 1.0 / math.sqrt(wl.d)
    state = {key: [cu_r, lens_r.astype(np.int64), Kf.copy(), Vf.copy()]
             for key, (cu_r, lens_r, Kf, Vf) in oracle_flat.items()}
    worst = 0.0
    for step in range(steps):
        dec = W.make_decode_batch(wl, step, tau, device="cuda", seqs=range(B), layers=range(L))
        out, code = run_decode(wl, shape, dec["q"], dec["k_new"], dec["v_new"], flat)
        assert code == 0
        o = np64(out)
        qn, kn, vn = np64(dec["q"]), np64(dec["k_new"]), np64(dec["v_new"])
        for b in range(B):
            for l in range(L):
                cu_r, lens_r, Kf, Vf = state[(b, l)]
                ref, Kn, Vn, ln = O.flat_decode(qn[b, l], Kf, Vf, cu_r, lens_r, scale,
                                                kn[b, l], vn[b, l])
                state[(b, l)] = [cu_r, ln, Kn, Vn]
                err = assert_decode_close(o[b, l], ref, wl.dtype, atol=atol,
                                          what="decode step %d b%d l%d" % (step, b, l))
                worst = max(worst, err)
    lens_gpu = flat["lens"].cpu().numpy()
    for (b, l), (_, ln, _, _) in state.items():
        np.testing.assert_array_equal(lens_gpu[b, l], ln)
    return worst


def full_check(wl, B=None, L=None, budgets=None, decode_steps=1, dec_atol=None):
    assert decode_steps <= wl.reserve, "each decode append needs a reserve row"
    B = wl.batch if B is None else B
    L = wl.layers if L is None else L
    shape = kv.KvShape.from_workload(wl, batch=B, layers=L)
    inp = W.make_batch(wl, device="cuda", seqs=range(B), layers=range(L))
    budgets = wl.budgets()[:B, :L] if (budgets is None and wl.budget_kind == "layer") else (
        wl.budgets()[:B] if budgets is None else budgets)
    scores, crit = run_score(wl, shape, inp)
    s_gpu = scores.cpu().numpy()
    c_gpu = crit.cpu().numpy() if crit is not None else None
    s_ref = np.zeros(s_gpu.shape)
    c_ref = np.zeros(s_gpu.shape) if crit is not None else None
    for b in range(B):
        for l in range(L):
            q, k, v, w_o = unit_np(inp, b, l, wl)
            s, c = oracle_scores(wl, q, k, v, w_o)
            s_ref[b, l] = s
            assert_scores_close(s_gpu[b, l].astype(np.float64), s, what="scores b%d l%d" % (b, l))
            if c is not None:
                c_ref[b, l] = c
                assert_scores_close(c_gpu[b, l].astype(np.float64), c,
                                    what="crit_norm b%d l%d" % (b, l))
    # end to end: GPU scores through GPU selection, against the oracle ranking
    lb, hb = run_allocate(wl, shape, scores, budgets)
    hbn = hb.cpu().numpy()
    assert np.all(hbn.sum(axis=2) == lb.cpu().numpy())
    cap = capacity_rows(wl, B, L, budgets)
    flat_e2e = run_compact(wl, shape, inp, scores, crit, hb, cap)
    kept = flat_e2e["kept"].cpu().numpy()
    cu = flat_e2e["cu"].cpu().numpy()
    for b in range(B):
        for l in range(L):
            for g in range(wl.hkv):
                k_g = int(hbn[b, l, g]) - wl.w
                base = cu[b, l, g]
                if crit is None:
                    oracle_kept_check(s_ref[b, l, g], kept[base:base + k_g], k_g)
                else:
                    oracle_crit_kept_check(s_ref[b, l, g], c_ref[b, l, g], s_gpu[b, l, g],
                                           kept[base:base + k_g], k_g, wl.crit_alpha[0],
                                           wl.crit_alpha[1], wl.crit_eps)
    # integer parity fed with the oracle's scores
    s32 = s_ref.astype(np.float32)
    c32 = c_ref.astype(np.float32) if c_ref is not None else None
    flat, oracle_flat = check_fed_oracle_scores(wl, shape, inp, s32, c32, budgets)
    worst = 0.0
    if decode_steps:
        tau = inp["tau"]
        atol = dec_atol if dec_atol is not None else (1e-2 if wl.dtype == "bf16" else 1e-4)
        worst = decode_and_check(wl, shape, flat, oracle_flat, decode_steps, tau, atol)
    return {"scores": s_gpu, "ref": s_ref, "decode_err": worst}


def test_tiny_mha_f32_full():
    full_check(W.WORKLOADS["tiny_mha_f32"].with_(reserve=2), decode_steps=2)


@pytest.mark.parametrize("frac", [0.2, 0.4, 0.8])
def test_llama_16k_layer(frac):
    wl = W.WORKLOADS["llama8b_16k_layer"].with_(head_budget_frac=frac)
    full_check(wl, decode_steps=3 if frac == 0.4 else 1)


def test_lava_entropy_layers_small():
    wl = W.WORKLOADS["mistral7b_128k_lava"].with_(n=4096, layers=4, reserve=4)
    full_check(wl, decode_steps=2)


def test_criticalkv_small():
    wl = W.WORKLOADS["llama8b_64k_criticalkv"].with_(n=2048, layers=2, model_dim=1024, reserve=2)
    full_check(wl, decode_steps=1)


def test_ada_batch_multi_layer_ragged():
    """Several sequences and layers, n not a multiple of any tile, G = 3, pool 3, d = 64."""
    wl = W.Workload(name="ragged", batch=2, layers=3, hq=6, hkv=2, d=64, n=1000 + 7, w=13, pool=3,
                    dtype="bf16", temp=(0.5, 16.0), head_budget_tokens=300, reserve=3,
                    seed=77)
    full_check(wl, decode_steps=2)


def test_ragged_f32_tiny_candidates():
    """C = 1: a single candidate per head."""
    wl = W.Workload(name="c1", batch=1, layers=2, hq=4, hkv=2, d=32, n=9, w=8, pool=7,
                    dtype="f32", temp=(0.5, 8.0), layer_budget=2 * 8 + 1, reserve=1, seed=5)
    full_check(wl, decode_steps=1)


def test_zero_selectable_budget_keeps_only_windows():
    wl = W.WORKLOADS["tiny_mha_f32"].with_(layer_budget=8 * 4)
    full_check(wl, decode_steps=1)


def test_full_budget_decode_equals_dense_attention():
    """B = n*Hkv keeps every row: flat decode (with one append) equals dense attention."""
    wl = W.Workload(name="full", batch=1, layers=2, hq=8, hkv=2, d=128, n=600, w=32, pool=7,
                    dtype="bf16", temp=(0.5, 16.0), layer_budget=600 * 2, reserve=1, seed=11)
    B, L = 1, 2
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    scores, _ = run_score(wl, shape, inp)
    budgets = wl.budgets()
    lb, hb = run_allocate(wl, shape, scores, budgets)
    assert torch.all(hb == wl.n)
    flat = run_compact(wl, shape, inp, scores, None, hb, capacity_rows(wl, B, L, budgets))
    dec = W.make_decode_batch(wl, 0, inp["tau"], device="cuda")
    out, code = run_decode(wl, shape, dec["q"], dec["k_new"], dec["v_new"], flat)
    assert code == 0
    o = np64(out)
    for l in range(L):
        K2 = np.concatenate([np64(inp["k"][0, l]), np64(dec["k_new"][0, l])[:, None]], axis=1)
        V2 = np.concatenate([np64(inp["v"][0, l]), np64(dec["v_new"][0, l])[:, None]], axis=1)
        ref = O.dense_decode(np64(dec["q"][0, l]), K2, V2, 1 / math.sqrt(wl.d))
        assert_decode_close(o[0, l], ref, wl.dtype, what="full-budget decode l%d" % l)


def test_all_tied_scores_follow_total_order():
    """Constant scores: every choice is a tie, decided by (head, position) order."""
    wl = W.Workload(name="ties", batch=1, layers=1, hq=8, hkv=4, d=64, n=300, w=16, pool=7,
                    dtype="bf16", temp=(1.0, 1.0), layer_budget=4 * 16 + 333, reserve=0, seed=3)
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    C = wl.n - wl.w
    s = np.full((1, 1, wl.hkv, C), 0.25, dtype=np.float32)
    s[0, 0, 2, 100:120] = 0.5
    check_fed_oracle_scores(wl, shape, inp, s, None, wl.budgets())


def test_decode_without_reserve_reports_device_check():
    wl = W.WORKLOADS["tiny_mha_f32"].with_(reserve=0)
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    scores, _ = run_score(wl, shape, inp)
    budgets = wl.budgets()
    lb, hb = run_allocate(wl, shape, scores, budgets)
    flat = run_compact(wl, shape, inp, scores, None, hb, capacity_rows(wl, 1, 1, budgets),
                       reserve=0)
    lens0 = flat["lens"].clone()
    dec = W.make_decode_batch(wl, 0, inp["tau"], device="cuda")
    out, code = run_decode(wl, shape, dec["q"], dec["k_new"], dec["v_new"], flat)
    assert code == 3            # no reserve row: the append is skipped
    assert torch.equal(flat["lens"], lens0)
    out2, code2 = run_decode(wl, shape, dec["q"], None, None, flat)
    assert code2 == 0
    assert torch.equal(out, out2)


def test_capacity_overflow_is_caught_and_bounded():
    wl = W.WORKLOADS["tiny_mha_f32"]
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    scores, _ = run_score(wl, shape, inp)
    lb, hb = run_allocate(wl, shape, scores, wl.budgets())
    cap = wl.hkv * (wl.w + wl.reserve) + 5
    guard = 64
    kept = torch.full((cap + guard,), -7, dtype=torch.int32, device="cuda")
    cu = torch.empty(1, 1, wl.hkv + 1, dtype=torch.int64, device="cuda")
    lens = torch.empty(1, 1, wl.hkv, dtype=torch.int32, device="cuda")
    kf = torch.full((cap + guard, wl.d), 3.0, dtype=torch.float32, device="cuda")
    vf = torch.full_like(kf, 3.0)
    from tests.kvpath import workspace
    ws = workspace(kv.KV_OP_COMPACT, shape)
    kv.kv_compact(shape, inp["k"], inp["v"], scores, None, 1, 2, 0.0, hb, wl.reserve, kept, cu,
                  lens, kf, vf, cap, ws)
    assert kv.kv_check_device_status(ws) == 2
    assert torch.all(kept[cap:] == -7)
    assert torch.all(kf[cap:] == 3.0) and torch.all(vf[cap:] == 3.0)


def test_out_of_range_budget_is_reported():
    wl = W.WORKLOADS["tiny_mha_f32"]
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    scores, _ = run_score(wl, shape, inp)
    from tests.kvpath import workspace
    ws = workspace(kv.KV_OP_ALLOCATE, shape)
    lb = torch.empty(1, 1, dtype=torch.int32, device="cuda")
    hb = torch.empty(1, 1, wl.hkv, dtype=torch.int32, device="cuda")
    bad = torch.tensor([[wl.w * wl.hkv - 1]], dtype=torch.int64, device="cuda")
    kv.kv_allocate(shape, scores, bad, 0, 1, 5, lb, hb, ws)
    assert kv.kv_check_device_status(ws) == 1
    assert int(lb) == wl.w * wl.hkv and torch.all(hb == wl.w)


def test_empty_batch_no_launch():
    wl = W.WORKLOADS["tiny_mha_f32"]
    shape = kv.KvShape.from_workload(wl, batch=0)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    kv.kv_score(shape, 0, 0, None, None, None, None, 0, None, None, ws)
    assert kv.kv_check_device_status(ws) == 0
