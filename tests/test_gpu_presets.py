"""Budget presets and re-eviction on the GPU against the oracle.

- StreamingLLM (4 sinks + the most recent rows, uniform per-head budgets from kv_allocate
  with alpha = 1): kept positions and gathered rows bit-exact against
  oracle.streaming_positions, and a decode step over the result within the decode bar;
- re-eviction during decoding: after decode steps have appended rows, kv_recompact shrinks
  every head; kept rows (appended and window rows always kept, prefill rows by their prefill
  scores) and their K/V bit-exact against oracle.reevict_rows, then a decode step.
"""
import math

import numpy as np
import pytest
import torch

import kv_cache_eviction_gb300 as kv
import oracle as O
from kv_cache_eviction_gb300 import workloads as W
from tests.kvpath import (assert_decode_close, capacity_rows, np64, run_allocate, run_compact,
                          run_decode, run_score, workspace)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_eviction_gb300 import _build
    _build.build()
    kv.lib()


def wl_small(**kw):
    base = dict(name="presets", batch=1, layers=2, hq=8, hkv=2, d=128, n=2000, w=32, pool=7,
                dtype="bf16", temp=(0.5, 16.0), head_budget_frac=0.25, reserve=6, seed=17)
    base.update(kw)
    return W.Workload(**base)


def check_decode(wl, shape, flat_np, dec, out):
    scale = 1.0 / math.sqrt(wl.d)
    cu, lens, Kf, Vf = flat_np
    for l in range(wl.layers):
        base, end = int(cu[l, 0]), int(cu[l, -1])
        ref, *_ = O.flat_decode(np64(dec["q"][0, l]), Kf[base:end], Vf[base:end], cu[l] - base,
                                lens[l].astype(np.int64), scale, np64(dec["k_new"][0, l]), np64(dec["v_new"][0, l]))
        assert_decode_close(np64(out[0, l]), ref, wl.dtype, what="decode l%d" % l)


def test_streaming_preset_matches_oracle():
    wl = wl_small(alpha=(1, 1))
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    scores, _ = run_score(wl, shape, inp)
    budgets = wl.budgets()
    _, hb = run_allocate(wl, shape, scores, budgets)           # alpha = 1: uniform budgets
    cap = capacity_rows(wl, 1, wl.layers, budgets)
    kept = torch.full((cap,), -7, dtype=torch.int32, device="cuda")
    cu = torch.empty(1, wl.layers, wl.hkv + 1, dtype=torch.int64, device="cuda")
    lens = torch.empty(1, wl.layers, wl.hkv, dtype=torch.int32, device="cuda")
    kf = torch.zeros(cap, wl.d, dtype=torch.bfloat16, device="cuda")
    vf = torch.zeros_like(kf)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    kv.kv_compact_streaming(shape, inp["k"], inp["v"], 4, hb, wl.reserve, kept, cu, lens, kf, vf,
                            cap, ws)
    assert kv.kv_check_device_status(ws) == 0
    C = wl.n - wl.w
    hbn, keptn, cun = hb.cpu().numpy(), kept.cpu().numpy(), cu.cpu().numpy()
    Kf, Vf = np64(kf), np64(vf)
    for l in range(wl.layers):
        K, V = np64(inp["k"][0, l]), np64(inp["v"][0, l])
        for g in range(wl.hkv):
            Bg = int(hbn[0, l, g]) - wl.w
            ref = np.concatenate([O.streaming_positions(C, Bg, 4), np.arange(C, wl.n)])
            r0 = cun[0, l, g]
            np.testing.assert_array_equal(keptn[r0:r0 + len(ref)], ref)
            assert np.all(keptn[r0 + len(ref):r0 + len(ref) + wl.reserve] == -1)
            np.testing.assert_array_equal(Kf[r0:r0 + len(ref)], K[g][ref])
            np.testing.assert_array_equal(Vf[r0:r0 + len(ref)], V[g][ref])
    flat_np = (cun[0].copy(), lens.cpu().numpy()[0].astype(np.int64), Kf.copy(), Vf.copy())
    dec = W.make_decode_batch(wl, 0, inp["tau"], device="cuda")
    out, code = run_decode(wl, shape, dec["q"], dec["k_new"], dec["v_new"],
                           {"kf": kf, "vf": vf, "cu": cu, "lens": lens})
    assert code == 0
    check_decode(wl, shape, flat_np, dec, out)


def test_reeviction_after_decode_appends():
    wl = wl_small()
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    scores, _ = run_score(wl, shape, inp)
    budgets = wl.budgets()
    _, hb = run_allocate(wl, shape, scores, budgets)
    cap = capacity_rows(wl, 1, wl.layers, budgets)
    flat = run_compact(wl, shape, inp, scores, None, hb, cap)
    steps = 4
    for st in range(steps):
        dec = W.make_decode_batch(wl, st, inp["tau"], device="cuda")
        _, code = run_decode(wl, shape, dec["q"], dec["k_new"], dec["v_new"], flat)
        assert code == 0
    # shrink every head by 37 prefill rows (its appended and window rows stay)
    lens_old = flat["lens"].clone()
    new_hb = (lens_old - 37).to(torch.int32)
    cap2 = int(new_hb.sum()) + wl.layers * wl.hkv * wl.reserve
    kept2 = torch.full((cap2,), -7, dtype=torch.int32, device="cuda")
    cu2 = torch.empty_like(flat["cu"])
    lens2 = torch.empty_like(flat["lens"])
    kf2 = torch.zeros(cap2, wl.d, dtype=torch.bfloat16, device="cuda")
    vf2 = torch.zeros_like(kf2)
    w_r = torch.zeros(kv.kv_recompact_workspace_size(cap), dtype=torch.uint8, device="cuda")
    kv.kv_recompact(shape, scores, new_hb, flat["kept"], flat["cu"], flat["lens"], flat["kf"],
                    flat["vf"], wl.reserve, None, kept2, cu2, lens2, kf2, vf2, w_r)
    assert kv.kv_check_device_status(w_r) == 0
    keptn, cun, lensn = flat["kept"].cpu().numpy(), flat["cu"].cpu().numpy(), lens_old.cpu().numpy()
    Kf, Vf = np64(flat["kf"]), np64(flat["vf"])
    kept2n, cu2n, Kf2, Vf2 = kept2.cpu().numpy(), cu2.cpu().numpy(), np64(kf2), np64(vf2)
    s32 = scores.cpu().numpy()
    np.testing.assert_array_equal(lens2.cpu().numpy(), new_hb.cpu().numpy())
    for l in range(wl.layers):
        for g in range(wl.hkv):
            r0, m = cun[0, l, g], lensn[0, l, g]
            held = keptn[r0:r0 + m]
            assert np.sum(held == -1) == steps                     # the appended rows
            rows = O.reevict_rows(held, s32[0, l, g].astype(np.float64), int(new_hb[0, l, g]))
            d0 = cu2n[0, l, g]
            np.testing.assert_array_equal(kept2n[d0:d0 + len(rows)], held[rows])
            np.testing.assert_array_equal(Kf2[d0:d0 + len(rows)], Kf[r0 + rows])
            np.testing.assert_array_equal(Vf2[d0:d0 + len(rows)], Vf[r0 + rows])
    flat_np = (cu2n[0].copy(), lens2.cpu().numpy()[0].astype(np.int64), Kf2.copy(), Vf2.copy())
    dec = W.make_decode_batch(wl, steps, inp["tau"], device="cuda")
    out, code = run_decode(wl, shape, dec["q"], dec["k_new"], dec["v_new"],
                           {"kf": kf2, "vf": vf2, "cu": cu2, "lens": lens2})
    assert code == 0
    check_decode(wl, shape, flat_np, dec, out)
