"""Nothing is written outside the buffers the calls are given.

Each output sits inside a larger allocation whose head and tail hold sentinel values; the
flat cache has rows past flat_capacity_rows; every workspace is kv_workspace_size bytes
followed by a sentinel tail.  After a full pass (kv_score, kv_allocate, kv_compact and a
few decode steps through each decode kernel) every sentinel must be untouched.
"""
import os

import pytest
import torch

import kv_cache_eviction_gb300 as kv
from kv_cache_eviction_gb300 import workloads as W
from tests.kvpath import GROUP, MODE, capacity_rows

pytestmark = pytest.mark.gpu

GUARD = 4096   # elements (or bytes, for workspaces) on each side


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_eviction_gb300 import _build
    _build.build()
    kv.lib()


class Guarded:
    """A tensor of `shape` inside a flat allocation with GUARD sentinel elements around it."""

    def __init__(self, shape, dtype, fill, sentinel):
        n = 1
        for s in shape:
            n *= s
        self.buf = torch.full((GUARD + n + GUARD,), sentinel, dtype=dtype, device="cuda")
        self.buf[GUARD:GUARD + n] = fill
        self.t = self.buf[GUARD:GUARD + n].view(*shape)
        self.sentinel = sentinel
        self.n = n

    def intact(self):
        head, tail = self.buf[:GUARD], self.buf[GUARD + self.n:]
        return bool((head == self.sentinel).all()) and bool((tail == self.sentinel).all())


def guarded_ws(op, shape):
    n = max(kv.kv_workspace_size(op, shape), 256)
    buf = torch.full((n + GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    buf[:n] = 0
    return buf, n


@pytest.mark.parametrize("path", [None, "split", "heads", "rows", "parts"])
@pytest.mark.parametrize("name,kw", [
    ("mistral7b_128k_lava", dict(layers=2, n=16384)),
    ("llama8b_64k_criticalkv", dict(layers=2, n=8192, model_dim=1024)),
])
def test_no_writes_outside_buffers(path, name, kw):
    old = os.environ.get("KVEVICT_DECODE_PATH")
    if path is None:
        os.environ.pop("KVEVICT_DECODE_PATH", None)
    else:
        os.environ["KVEVICT_DECODE_PATH"] = path
    try:
        wl = W.WORKLOADS[name].with_(**kw)
        shape = kv.KvShape.from_workload(wl)
        B, L, C = wl.batch, wl.layers, wl.n - wl.w
        inp = W.make_batch(wl, device="cuda")
        budgets = wl.budgets().cuda()
        cap = capacity_rows(wl, B, L, wl.budgets())
        scores = Guarded((B, L, wl.hkv, C), torch.float32, 0.0, -123.0)
        crit = Guarded((B, L, wl.hkv, C), torch.float32, 0.0, -123.0) \
            if wl.mode == "critical" else None
        lb = Guarded((B, L), torch.int32, 0, -77)
        hb = Guarded((B, L, wl.hkv), torch.int32, 0, -77)
        kept = Guarded((cap,), torch.int32, 0, -77)
        cu = Guarded((B, L, wl.hkv + 1), torch.int64, 0, -77)
        lens = Guarded((B, L, wl.hkv), torch.int32, 0, -77)
        # flat cache rows past `cap` belong to nobody: appends must stop at the capacity
        kf = Guarded((cap + 64, wl.d), wl.torch_dtype, 0.0, 7.0)
        vf = Guarded((cap + 64, wl.d), wl.torch_dtype, 0.0, 7.0)
        kf.t[cap:] = 7.0
        vf.t[cap:] = 7.0
        ws = {op: guarded_ws(op, shape) for op in (kv.KV_OP_SCORE, kv.KV_OP_ALLOCATE,
                                                   kv.KV_OP_COMPACT, kv.KV_OP_DECODE)}

        def wsv(op):
            buf, n = ws[op]
            return buf[:n]

        kv.kv_score(shape, MODE[wl.mode], GROUP[wl.group], inp["q_win"], inp["k"],
                    inp["v"] if wl.mode != "ada" else None, inp.get("w_o"), wl.model_dim,
                    scores.t, crit.t if crit else None, wsv(kv.KV_OP_SCORE))
        kv.kv_allocate(shape, scores.t, budgets, 1 if wl.budget_kind == "total" else 0,
                       wl.alpha[0], wl.alpha[1], lb.t, hb.t, wsv(kv.KV_OP_ALLOCATE))
        kv.kv_compact(shape, inp["k"], inp["v"], scores.t, crit.t if crit else None,
                      wl.crit_alpha[0], wl.crit_alpha[1], wl.crit_eps, hb.t, wl.reserve,
                      kept.t, cu.t, lens.t, kf.t, vf.t, cap, wsv(kv.KV_OP_COMPACT))
        outs = []
        for s_ in range(3):
            dec = W.make_decode_batch(wl, s_, inp["tau"], device="cuda")
            out = Guarded(tuple(dec["q"].shape), wl.torch_dtype, 0.0, 5.0)
            kv.flat_decode_attn(shape, dec["q"], dec["k_new"], dec["v_new"], kf.t, vf.t, cu.t,
                                lens.t, 1.0 / wl.d ** 0.5, out.t, wsv(kv.KV_OP_DECODE),
                                flat_capacity_rows=cap)
            outs.append(out)
        torch.cuda.synchronize()
        for op in ws:
            assert kv.kv_check_device_status(wsv(op)) == 0
        for nm, g in [("scores", scores), ("crit", crit), ("layer budgets", lb),
                      ("head budgets", hb), ("kept", kept), ("cu", cu), ("lens", lens)]:
            if g is not None:
                assert g.intact(), nm
        # the flat cache: the guards around the allocation and every row past cap
        for nm, g in [("k_flat", kf), ("v_flat", vf)]:
            assert g.intact(), nm
            assert bool((g.t[cap:] == 7.0).all()), nm + " rows past the capacity"
        for i, o in enumerate(outs):
            assert o.intact(), "decode output %d" % i
        for op, (buf, n) in ws.items():
            assert bool((buf[n:] == 0xA5).all()), "workspace tail of op %d" % op
    finally:
        if old is None:
            os.environ.pop("KVEVICT_DECODE_PATH", None)
        else:
            os.environ["KVEVICT_DECODE_PATH"] = old


def test_next_calls_write_nothing_outside_their_buffers():
    """The same sentinels around the outputs of the cascade's calls (capped allocation,
    re-compaction from a flat cache and from the K/V at a device-side row base), the
    per-query-head terms and scores, the two-stage compaction with kappa given, the
    StreamingLLM preset and the model-wide allocation."""
    import math
    wl = W.WORKLOADS["mistral7b_128k_lava"].with_(layers=3, n=6000)
    shape = kv.KvShape.from_workload(wl)
    B, L, C, hkv, hq = 1, wl.layers, wl.n - wl.w, wl.hkv, wl.hq
    inp = W.make_batch(wl, device="cuda")
    scores = Guarded((B, L, hkv, C), torch.float32, 0.0, -123.0)
    ws_s, n_s = guarded_ws(kv.KV_OP_SCORE, shape)
    kv.kv_score(shape, kv.KV_SCORE_LAVA, kv.KV_GROUP_MAX, inp["q_win"], inp["k"], inp["v"],
                None, 0, scores.t, None, ws_s[:n_s])
    total = wl.total_budget_value()
    cap = total + L * hkv * 2
    caps = Guarded((B, L), torch.int32, wl.n * hkv, -77)
    lb = Guarded((B, L), torch.int32, 0, -77)
    hb = Guarded((B, L, hkv), torch.int32, 0, -77)
    ws_a, n_a = guarded_ws(kv.KV_OP_ALLOCATE, shape)
    kv.kv_allocate_capped(shape, scores.t, torch.tensor([total], dtype=torch.int64,
                                                        device="cuda"),
                          caps.t, 0, 1, lb.t, hb.t, ws_a[:n_a])
    flats = []
    for _ in range(2):
        flats.append({"kept": Guarded((cap,), torch.int32, -5, -77),
                      "cu": Guarded((B, L, hkv + 1), torch.int64, 0, -77),
                      "lens": Guarded((B, L, hkv), torch.int32, 0, -77),
                      "kf": Guarded((cap, wl.d), wl.torch_dtype, 0.0, 7.0),
                      "vf": Guarded((cap, wl.d), wl.torch_dtype, 0.0, 7.0)})
    nr = kv.kv_recompact_workspace_size(max(cap, L * hkv * wl.n))
    wr = torch.full((nr + GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    wr[:nr] = 0
    f0, f1 = flats
    # layers 0..L-2 from the K/V, then layer L-1 at the row base the first call ends at
    sh0 = kv.KvShape.from_workload(wl, layers=L - 1)
    kv.kv_recompact(sh0, scores.t[:, :L - 1], hb.t[:, :L - 1].contiguous(), None, None, None,
                    inp["k"][:, :L - 1], inp["v"][:, :L - 1], 2, None, f0["kept"].t,
                    f0["cu"].t, f0["lens"].t, f0["kf"].t, f0["vf"].t, wr[:nr])
    kv.kv_recompact(kv.KvShape.from_workload(wl, layers=1), scores.t[:, L - 1:],
                    hb.t[:, L - 1:].contiguous(), None, None, None, inp["k"][:, L - 1:],
                    inp["v"][:, L - 1:], 2, f0["cu"].t[0, L - 2, hkv:hkv + 1], f0["kept"].t,
                    f0["cu"].t[:, L - 1:], f0["lens"].t[:, L - 1:], f0["kf"].t, f0["vf"].t,
                    wr[:nr])
    # then every head 10 rows smaller, from that flat cache into the other
    new_hb = (f0["lens"].t - 10).clamp(min=wl.w).to(torch.int32).contiguous()
    kv.kv_recompact(shape, scores.t, new_hb, f0["kept"].t, f0["cu"].t, f0["lens"].t, f0["kf"].t,
                    f0["vf"].t, 2, None, f1["kept"].t, f1["cu"].t, f1["lens"].t, f1["kf"].t,
                    f1["vf"].t, wr[:nr])
    # StreamingLLM preset into the first buffer again
    kv.kv_compact_streaming(shape, inp["k"], inp["v"], 4, hb.t, 2, f0["kept"].t, f0["cu"].t,
                            f0["lens"].t, f0["kf"].t, f0["vf"].t, cap, ws_s[:256])
    # per-query-head terms and scores (W_O per query head), kappa compaction, model-wide
    D = 520
    w_oq = (torch.randn(L, hq, wl.d, D, device="cuda") / math.sqrt(D)).to(torch.bfloat16)
    terms = Guarded((B, L, hq, C), torch.float32, 0.0, -123.0)
    proj = Guarded((B, L, hkv, C), torch.float32, 0.0, -123.0)
    outs = []
    for tk, pk in ((kv.KV_TERMS_MEAN_POOLED, kv.KV_PROJ_CRIT_GQA), (kv.KV_TERMS_L2,
                                                                      kv.KV_PROJ_LAPROX)):
        kv.kv_window_terms(shape, tk, inp["q_win"], inp["k"], terms.t, ws_s[:n_s])
        kv.kv_proj_score(shape, pk, inp["v"], w_oq, D, terms.t, 1e-3, proj.t, ws_s[:256])
    ws_c, n_c = guarded_ws(kv.KV_OP_COMPACT, shape)
    kv.kv_compact_kappa(shape, inp["k"], inp["v"], scores.t, proj.t, 1, 2, hb.t, 2,
                        f1["kept"].t, f1["cu"].t, f1["lens"].t, f1["kf"].t, f1["vf"].t, cap,
                        ws_c[:n_c])
    kv.kv_allocate(shape, proj.t, torch.tensor([total], dtype=torch.int64, device="cuda"), 2,
                   0, 1, lb.t, hb.t, ws_a[:n_a])
    torch.cuda.synchronize()
    for buf, n in ((ws_s, n_s), (ws_a, n_a), (ws_c, n_c)):
        assert kv.kv_check_device_status(buf[:n]) == 0
        assert bool((buf[n:] == 0xA5).all())
    assert kv.kv_check_device_status(wr[:nr]) == 0
    assert bool((wr[nr:] == 0xA5).all()), "recompaction workspace tail"
    for nm, g in [("scores", scores), ("caps", caps), ("lb", lb), ("hb", hb), ("terms", terms),
                  ("proj", proj)]:
        assert g.intact(), nm
    for i, f in enumerate(flats):
        for nm, g in f.items():
            assert g.intact(), "flat %d %s" % (i, nm)
