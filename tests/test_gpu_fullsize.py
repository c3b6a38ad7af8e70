"""Full-size parity on sampled units.

The three multi-layer workloads run at their full sizes through the same calls bench.py
times (kv_score, kv_allocate and kv_compact over every (sequence, layer) of the batch, then
one flat_decode_attn step over all of them).  The oracle then checks four (sequence,
layer) units, always including the first and the last:

- scores within 1e-4 relative of the oracle's fp64 scores of that unit (CriticalKV: the
  ||(V W_O)_j||_1 norms on a seeded sample of rows, the full product being 275 GFLOP per
  layer in fp64);
- budgets, kept indices, offsets and gathered rows bit-exact against the oracle fed the
  GPU's own float32 scores (LAVa layer budgets from the entropies of all layers);
- the decode step of the unit within the decode tolerance of the oracle run on the GPU's
  flat cache of that unit.
"""
import math

import numpy as np
import pytest
import torch

import kv_cache_eviction_gb300 as kv
import oracle as O
from kv_cache_eviction_gb300 import workloads as W
from tests.kvpath import (assert_decode_close, assert_scores_close, capacity_rows, np64,
                          run_allocate, run_compact, run_decode, run_score)
from tests.test_gpu_parity import oracle_scores

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_eviction_gb300 import _build
    _build.build()
    kv.lib()


def samples(B, L, seed, n=4):
    """n distinct (sequence, layer) units: the first, the last, and seeded interior layers."""
    rng = np.random.default_rng(seed)
    pts = [(0, 0), (B - 1, L - 1)]
    while len(pts) < n:
        p = (int(rng.integers(B)), int(rng.integers(1, L - 1)))
        if p not in pts:
            pts.append(p)
    return pts


@pytest.mark.parametrize("name", ["llama8b_32k_b4", "mistral7b_128k_lava",
                                  "llama8b_64k_criticalkv"])
def test_fullsize_sampled_units(name):
    wl = W.WORKLOADS[name]
    B, L, hkv = wl.batch, wl.layers, wl.hkv
    C = wl.n - wl.w
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    budgets = wl.budgets()
    scores, crit = run_score(wl, shape, inp)
    lb, hb = run_allocate(wl, shape, scores, budgets)
    cap = capacity_rows(wl, B, L, budgets)
    flat = run_compact(wl, shape, inp, scores, crit, hb, cap)
    torch.cuda.synchronize()
    s32 = scores.cpu().numpy()
    c32 = crit.cpu().numpy() if crit is not None else None
    lb_h, hb_h = lb.cpu().numpy(), hb.cpu().numpy()
    cu_h, lens_h = flat["cu"].cpu().numpy(), flat["lens"].cpu().numpy()
    a, b_ = wl.alpha

    # layer budgets of every sequence, from the GPU's scores
    for bb in range(B):
        if wl.budget_kind == "total":
            e = [O.layer_entropy(s32[bb, l].astype(np.float64), wl.n) for l in range(L)]
            ref = O.lava_layer_budgets(e, int(budgets[bb]), wl.w, hkv, C)
        else:
            ref = budgets[bb].numpy()
        np.testing.assert_array_equal(lb_h[bb], ref)

    pts = samples(B, L, seed=len(name))
    for (bb, l) in pts:
        k = np64(inp["k"][bb, l])
        v = np64(inp["v"][bb, l])
        q = np64(inp["q_win"][bb, l])
        # scores of the unit (CriticalKV: its A scores; the norms are sampled below)
        s_ref, _ = oracle_scores(wl, q, k, v, None, mode="ada" if wl.mode == "critical"
                                 else wl.mode)
        assert_scores_close(s32[bb, l].astype(np.float64), s_ref, what="scores %d/%d" % (bb, l))
        if c32 is not None:
            rng = np.random.default_rng(bb * 1000 + l)
            w_o = np64(inp["w_o"][l])
            for g in range(hkv):
                rows = np.sort(rng.choice(C, size=256, replace=False))
                ref = O.critical_row_norm(v[g:g + 1, rows], w_o[g:g + 1], len(rows))[0]
                assert_scores_close(c32[bb, l, g, rows].astype(np.float64), ref,
                                    what="crit %d/%d/%d" % (bb, l, g))
        # integer outputs, the oracle fed the GPU's float32 scores
        s64 = s32[bb, l].astype(np.float64)
        f, Bg = O.head_budgets(s64, int(lb_h[bb, l]), wl.w, a, b_)
        np.testing.assert_array_equal(hb_h[bb, l], Bg + wl.w)
        cr = None
        c64 = None
        if c32 is not None:
            cr = (wl.crit_alpha[0], wl.crit_alpha[1], wl.crit_eps)
            c64 = c32[bb, l].astype(np.float64)
        kept_r, cu_r, lens_r, Kf, Vf = O.compact_layer(k, v, s64, Bg, wl.w, reserve=wl.reserve,
                                                       c=c64, crit=cr, kappa_dtype=np.float32)
        base = int(cu_h[bb, l, 0])
        np.testing.assert_array_equal(cu_h[bb, l] - base, cu_r)
        np.testing.assert_array_equal(lens_h[bb, l], lens_r)
        end = int(cu_h[bb, l, -1])
        kept_seg = flat["kept"][base:end].cpu().numpy()
        kf_seg = np64(flat["kf"][base:end])
        vf_seg = np64(flat["vf"][base:end])
        for g in range(hkv):
            r0 = cu_r[g]
            np.testing.assert_array_equal(kept_seg[r0:r0 + lens_r[g]], kept_r[g])
            np.testing.assert_array_equal(kf_seg[r0:r0 + lens_r[g]], Kf[r0:r0 + lens_r[g]])
            np.testing.assert_array_equal(vf_seg[r0:r0 + lens_r[g]], Vf[r0:r0 + lens_r[g]])

    # one decode step over every layer (with the append), checked on the sampled units
    segs = {}
    for (bb, l) in pts:
        base, end = int(cu_h[bb, l, 0]), int(cu_h[bb, l, -1])
        segs[(bb, l)] = (cu_h[bb, l] - base, lens_h[bb, l].astype(np.int64),
                         np64(flat["kf"][base:end]), np64(flat["vf"][base:end]))
    dec = W.make_decode_batch(wl, 0, inp["tau"], device="cuda")
    out, code = run_decode(wl, shape, dec["q"], dec["k_new"], dec["v_new"], flat)
    assert code == 0
    scale = 1.0 / math.sqrt(wl.d)
    for (bb, l), (cu_r, lens_r, Kf, Vf) in segs.items():
        ref, _, _, ln = O.flat_decode(np64(dec["q"][bb, l]), Kf, Vf, cu_r, lens_r, scale,
                                      np64(dec["k_new"][bb, l]), np64(dec["v_new"][bb, l]))
        o = np64(out[bb, l])
        assert_decode_close(o, ref, wl.dtype, what="decode %d/%d" % (bb, l))
        np.testing.assert_array_equal(flat["lens"][bb, l].cpu().numpy(), ln)
