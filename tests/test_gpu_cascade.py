"""LAVa's online layer-wise prefill cascade on the GPU against the oracle, stage by stage.

Stage t: kv_allocate_capped splits the sequence's total over layers 0..t-1 with each earlier
layer capped at what it holds; kv_recompact re-selects layers 0..t-2 from the previous flat
cache into a second buffer, then compacts the new layer t-1 from its uncompacted K/V right
after them (its row base read on the device from the first call's last offset).  Layer and
head budgets, offsets, lengths, kept positions and the gathered rows must be bit-exact
against the oracle's cascade fed the GPU's own float32 scores; a decode step over the final
cache must match the oracle's within the decode bar.
"""
import math

import numpy as np
import pytest
import torch

import kv_cache_eviction_gb300 as kv
import oracle as O
from kv_cache_eviction_gb300 import workloads as W
from tests.kvpath import assert_decode_close, np64, run_score

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_eviction_gb300 import _build
    _build.build()
    kv.lib()


def zeros_u8(nbytes):
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device="cuda")


def run_cascade(wl, total, reserve=2):
    """Runs the cascade through the C ABI; returns per-stage GPU results and the inputs."""
    L, hkv, n, w = wl.layers, wl.hkv, wl.n, wl.w
    C = n - w
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    scores, _ = run_score(wl, shape, inp)          # per layer; independent of the order
    cap_rows = total + L * hkv * reserve
    flats = []
    for _ in range(2):
        flats.append({"kept": torch.full((cap_rows,), -7, dtype=torch.int32, device="cuda"),
                      "cu": torch.zeros(1, L, hkv + 1, dtype=torch.int64, device="cuda"),
                      "lens": torch.zeros(1, L, hkv, dtype=torch.int32, device="cuda"),
                      "kf": torch.zeros(cap_rows, wl.d, dtype=wl.torch_dtype, device="cuda"),
                      "vf": torch.zeros(cap_rows, wl.d, dtype=wl.torch_dtype, device="cuda")})
    caps = [torch.full((1, L), n * hkv, dtype=torch.int32, device="cuda") for _ in range(2)]
    hb_all = torch.zeros(1, L, hkv, dtype=torch.int32, device="cuda")
    budget = torch.tensor([total], dtype=torch.int64, device="cuda")
    w_a = zeros_u8(kv.kv_workspace_size(kv.KV_OP_ALLOCATE, shape))
    w_r = zeros_u8(kv.kv_recompact_workspace_size(max(cap_rows, hkv * n)))
    stages = []
    for t in range(1, L + 1):
        sh_t = kv.KvShape.from_workload(wl, layers=t)
        lb = caps[t % 2]
        hb = torch.zeros(1, t, hkv, dtype=torch.int32, device="cuda")
        # caps: the previous stage's budgets for layers 0..t-2, the initial n*Hkv for t-1
        kv.kv_allocate_capped(sh_t, scores[:, :t], budget, caps[(t - 1) % 2], 0, 1, lb, hb, w_a)
        assert kv.kv_check_device_status(w_a) == 0
        src, dst = flats[(t - 1) % 2], flats[t % 2]
        dst["kept"].fill_(-7)
        if t >= 2:
            sh_old = kv.KvShape.from_workload(wl, layers=t - 1)
            kv.kv_recompact(sh_old, scores[:, :t - 1], hb[:, :t - 1].contiguous(), src["kept"],
                            src["cu"][:, :t - 1].contiguous(), src["lens"][:, :t - 1].contiguous(),
                            src["kf"], src["vf"], reserve, None, dst["kept"], dst["cu"],
                            dst["lens"], dst["kf"], dst["vf"], w_r)
            assert kv.kv_check_device_status(w_r) == 0
        sh_new = kv.KvShape.from_workload(wl, layers=1)
        row_base = dst["cu"][0, t - 2, hkv:hkv + 1] if t >= 2 else None
        kv.kv_recompact(sh_new, scores[:, t - 1:t].contiguous(), hb[:, t - 1:t].contiguous(),
                        None, None, None, inp["k"][:, t - 1:t].contiguous(),
                        inp["v"][:, t - 1:t].contiguous(), reserve, row_base, dst["kept"],
                        dst["cu"][:, t - 1:t], dst["lens"][:, t - 1:t], dst["kf"], dst["vf"], w_r)
        assert kv.kv_check_device_status(w_r) == 0
        torch.cuda.synchronize()
        stages.append({"layer_budget": lb[0, :t].cpu().numpy().copy(),
                       "head_budget": hb[0].cpu().numpy().copy(),
                       "cu": dst["cu"][0, :t].cpu().numpy().copy(),
                       "lens": dst["lens"][0, :t].cpu().numpy().copy(),
                       "kept": dst["kept"].cpu().numpy().copy(),
                       "kf": np64(dst["kf"]), "vf": np64(dst["vf"])})
    return inp, scores, stages, flats[L % 2]


@pytest.mark.parametrize("total_extra", [600, 2500])
def test_cascade_matches_oracle_stage_by_stage(total_extra):
    wl = W.Workload(name="cascade", batch=1, layers=4, hq=8, hkv=2, d=128, n=1500, w=16, pool=7,
                    dtype="bf16", temp=(0.5, 16.0), mode="lava", group="max",
                    budget_kind="total", alpha=(0, 1), reserve=2, seed=41)
    L, hkv, n, w = wl.layers, wl.hkv, wl.n, wl.w
    C = n - w
    total = 4 * w * hkv + total_extra
    reserve = 2
    inp, scores, stages, final = run_cascade(wl, total, reserve)
    S = [scores[0, l].double().cpu().numpy() for l in range(L)]
    ref = O.lava_cascade(S, total, w, n)
    K = [np64(inp["k"][0, l]) for l in range(L)]
    V = [np64(inp["v"][0, l]) for l in range(L)]
    for t, (got, x) in enumerate(zip(stages, ref), start=1):
        np.testing.assert_array_equal(got["layer_budget"], x["layer_budget"])
        np.testing.assert_array_equal(got["head_budget"], x["head_budget"])
        np.testing.assert_array_equal(got["lens"], x["head_budget"])
        row = 0
        for l in range(t):
            for g in range(hkv):
                assert got["cu"][l, g] == row
                kept = x["kept"][l][g]
                r0, r1 = row, row + len(kept)
                np.testing.assert_array_equal(got["kept"][r0:r1], kept)
                assert np.all(got["kept"][r1:r1 + reserve] == -1)
                np.testing.assert_array_equal(got["kf"][r0:r1], K[l][g][kept])
                np.testing.assert_array_equal(got["vf"][r0:r1], V[l][g][kept])
                row = r1 + reserve
            assert got["cu"][l, hkv] == row
    # a decode step over the final cache
    shape = kv.KvShape.from_workload(wl)
    dec = W.make_decode_batch(wl, 0, inp["tau"], device="cuda")
    out = torch.empty_like(dec["q"])
    wsd = zeros_u8(kv.kv_workspace_size(kv.KV_OP_DECODE, shape))
    kv.flat_decode_attn(shape, dec["q"], dec["k_new"], dec["v_new"], final["kf"], final["vf"],
                        final["cu"], final["lens"], 1.0 / math.sqrt(wl.d), out, wsd)
    assert kv.kv_check_device_status(wsd) == 0
    last = stages[-1]
    for l in range(L):
        base = int(last["cu"][l, 0])
        cu_l = last["cu"][l] - base
        end = int(last["cu"][l, hkv])
        o_ref, *_ = O.flat_decode(np64(dec["q"][0, l]), last["kf"][base:end], last["vf"][base:end],
                                  cu_l, last["lens"][l].astype(np.int64), 1.0 / math.sqrt(wl.d),
                                  np64(dec["k_new"][0, l]), np64(dec["v_new"][0, l]))
        assert_decode_close(np64(out[0, l]), o_ref, "bf16", what="cascade decode l%d" % l)


def test_recompact_from_full_kv_equals_kv_compact():
    """The uncompacted K/V as the source: kv_recompact gives kv_compact's flat cache."""
    from tests.kvpath import capacity_rows, run_allocate, run_compact
    wl = W.WORKLOADS["llama8b_16k_layer"].with_(n=3000, layers=2, reserve=3)
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    scores, _ = run_score(wl, shape, inp)
    budgets = wl.budgets()
    _, hb = run_allocate(wl, shape, scores, budgets)
    cap = capacity_rows(wl, 1, wl.layers, budgets)
    ref = run_compact(wl, shape, inp, scores, None, hb, cap)
    kept = torch.full((cap,), -7, dtype=torch.int32, device="cuda")
    cu = torch.zeros_like(ref["cu"])
    lens = torch.zeros_like(ref["lens"])
    kf = torch.zeros_like(ref["kf"])
    vf = torch.zeros_like(ref["vf"])
    w_r = zeros_u8(kv.kv_recompact_workspace_size(wl.layers * wl.hkv * wl.n))
    kv.kv_recompact(shape, scores, hb, None, None, None, inp["k"], inp["v"], wl.reserve, None,
                    kept, cu, lens, kf, vf, w_r)
    assert kv.kv_check_device_status(w_r) == 0
    for a, b in ((kept, ref["kept"]), (cu, ref["cu"]), (lens, ref["lens"]), (kf, ref["kf"]),
                 (vf, ref["vf"])):
        assert torch.equal(a, b)
