"""The path captured once as a CUDA graph and replayed gives what eager launches give.

bench.py times the step (kv_score, kv_allocate, kv_compact, flat_decode_attn) as a captured
graph and the decode alone as a captured graph of the call.  Every kernel of the path
reduces in a fixed order (partials by index, tickets merged by slot, histograms of integers),
so a replay must reproduce the eager outputs bit for bit: scores, budgets, kept indices,
offsets, lengths, the flat cache and the decode output.  The step is idempotent: compaction
rewrites the flat cache and the lengths before the decode appends to them.
"""
import os

import pytest
import torch

import kv_cache_eviction_gb300 as kv
from kv_cache_eviction_gb300 import workloads as W
from tests.kvpath import GROUP, MODE, capacity_rows, workspace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_eviction_gb300 import _build
    _build.build()
    kv.lib()


def make_step(wl):
    dev = torch.device("cuda")
    shape = kv.KvShape.from_workload(wl)
    B, L, C = wl.batch, wl.layers, wl.n - wl.w
    inp = W.make_batch(wl, device=dev)
    budgets = wl.budgets().to(dev)
    dec = W.make_decode_batch(wl, 0, inp["tau"], device=dev)
    cap = capacity_rows(wl, B, L, wl.budgets())
    ws = {op: workspace(op, shape) for op in (kv.KV_OP_SCORE, kv.KV_OP_ALLOCATE,
                                              kv.KV_OP_COMPACT, kv.KV_OP_DECODE)}
    o = {
        "scores": torch.empty(B, L, wl.hkv, C, dtype=torch.float32, device=dev),
        "lb": torch.empty(B, L, dtype=torch.int32, device=dev),
        "hb": torch.empty(B, L, wl.hkv, dtype=torch.int32, device=dev),
        "kept": torch.full((cap,), -7, dtype=torch.int32, device=dev),
        "cu": torch.empty(B, L, wl.hkv + 1, dtype=torch.int64, device=dev),
        "lens": torch.empty(B, L, wl.hkv, dtype=torch.int32, device=dev),
        "kf": torch.zeros(cap, wl.d, dtype=wl.torch_dtype, device=dev),
        "out": torch.empty_like(dec["q"]),
    }
    o["crit"] = torch.empty_like(o["scores"]) if wl.mode == "critical" else None
    o["vf"] = torch.zeros_like(o["kf"])
    entropy = 1 if wl.budget_kind == "total" else 0

    def step(st):
        kv.kv_score(shape, MODE[wl.mode], GROUP[wl.group], inp["q_win"], inp["k"],
                    inp["v"] if wl.mode != "ada" else None, inp.get("w_o"), wl.model_dim,
                    o["scores"], o["crit"], ws[kv.KV_OP_SCORE], st)
        kv.kv_allocate(shape, o["scores"], budgets, entropy, wl.alpha[0], wl.alpha[1], o["lb"],
                       o["hb"], ws[kv.KV_OP_ALLOCATE], st)
        kv.kv_compact(shape, inp["k"], inp["v"], o["scores"], o["crit"], wl.crit_alpha[0],
                      wl.crit_alpha[1], wl.crit_eps, o["hb"], wl.reserve, o["kept"], o["cu"],
                      o["lens"], o["kf"], o["vf"], cap, ws[kv.KV_OP_COMPACT], st)
        kv.flat_decode_attn(shape, dec["q"], dec["k_new"], dec["v_new"], o["kf"], o["vf"],
                            o["cu"], o["lens"], 1.0 / wl.d ** 0.5, o["out"],
                            ws[kv.KV_OP_DECODE], st)

    def check_status():
        for w_ in ws.values():
            assert kv.kv_check_device_status(w_) == 0

    return step, o, check_status


@pytest.mark.parametrize("name,kw", [
    ("mistral7b_128k_lava", dict(layers=2)),
    ("llama8b_32k_b4", dict(layers=2, batch=2)),
    ("llama8b_64k_criticalkv", dict(layers=2, n=8192, model_dim=1024)),
])
@pytest.mark.parametrize("path", [None, "split", "rows", "parts"])
def test_graph_replay_matches_eager(name, kw, path):
    old = os.environ.get("KVEVICT_DECODE_PATH")
    if path is None:
        os.environ.pop("KVEVICT_DECODE_PATH", None)
    else:
        os.environ["KVEVICT_DECODE_PATH"] = path
    try:
        wl = W.WORKLOADS[name].with_(**kw)
        step, o, check_status = make_step(wl)
        stream = torch.cuda.current_stream()
        step(stream)                      # eager (also the one-time kernel set-up)
        torch.cuda.synchronize()
        check_status()
        eager = {k: v.clone() for k, v in o.items() if v is not None}
        gs = torch.cuda.Stream()
        gs.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            step(gs)
        for _ in range(2):
            # the replay has to write these again (every entry of each)
            for k in ("scores", "crit", "out"):
                if o[k] is not None:
                    o[k].fill_(float("nan"))
            for k in ("lb", "hb", "cu", "lens"):
                o[k].fill_(-1)
            with torch.cuda.stream(gs):
                graph.replay()
            torch.cuda.synchronize()
            check_status()
            for k, v in eager.items():
                assert torch.equal(o[k], v), k
    finally:
        if old is None:
            os.environ.pop("KVEVICT_DECODE_PATH", None)
        else:
            os.environ["KVEVICT_DECODE_PATH"] = old


def test_next_paths_replay_bit_for_bit():
    """A cascade stage (capped allocation, re-compaction from a flat cache, the new layer at
    a device-side row base) and the LaProx path (L2 window terms, per-query-head projected
    scores, model-wide allocation, compaction) captured once and replayed: the same outputs
    as eager launches."""
    import math
    dev = torch.device("cuda")
    wl = W.WORKLOADS["mistral7b_128k_lava"].with_(layers=3, n=5000)
    shape = kv.KvShape.from_workload(wl)
    B, L, C, hkv, hq = 1, wl.layers, wl.n - wl.w, wl.hkv, wl.hq
    inp = W.make_batch(wl, device=dev)
    scores = torch.empty(B, L, hkv, C, device=dev)
    kv.kv_score(shape, kv.KV_SCORE_LAVA, kv.KV_GROUP_MAX, inp["q_win"], inp["k"], inp["v"], None,
                0, scores, None, workspace(kv.KV_OP_SCORE, shape))
    total = wl.total_budget_value()
    cap = total + L * hkv * 2
    D = 264
    w_oq = (torch.randn(L, hq, wl.d, D, device=dev) / math.sqrt(D)).to(torch.bfloat16)
    prev = {"kept": torch.full((cap,), -7, dtype=torch.int32, device=dev),
            "cu": torch.zeros(B, L, hkv + 1, dtype=torch.int64, device=dev),
            "lens": torch.zeros(B, L, hkv, dtype=torch.int32, device=dev),
            "kf": torch.zeros(cap, wl.d, dtype=torch.bfloat16, device=dev),
            "vf": torch.zeros(cap, wl.d, dtype=torch.bfloat16, device=dev)}
    # a previous stage (layers 0..L-2 from their K/V) to re-compact from
    # (the previous stage's own budgets: layer-wide top selections, so the next stage's
    # per-head budgets fit in what each head holds)
    sh_old = kv.KvShape.from_workload(wl, layers=L - 1)
    lb0 = torch.empty(B, L - 1, dtype=torch.int32, device=dev)
    hb0 = torch.empty(B, L - 1, hkv, dtype=torch.int32, device=dev)
    kv.kv_allocate(sh_old, scores[:, :L - 1], torch.tensor([total], dtype=torch.int64,
                                                         device=dev),
                   1, 0, 1, lb0, hb0, workspace(kv.KV_OP_ALLOCATE, sh_old))
    kv.kv_recompact(sh_old, scores[:, :L - 1], hb0, None, None, None, inp["k"][:, :L - 1],
                    inp["v"][:, :L - 1], 2, None, prev["kept"], prev["cu"], prev["lens"],
                    prev["kf"], prev["vf"],
                    torch.zeros(kv.kv_recompact_workspace_size((L - 1) * hkv * wl.n),
                                dtype=torch.uint8, device=dev))
    caps = torch.full((B, L), wl.n * hkv, dtype=torch.int32, device=dev)
    caps[0, :L - 1] = lb0[0]
    ws_a = workspace(kv.KV_OP_ALLOCATE, shape)
    ws_s = workspace(kv.KV_OP_SCORE, shape)
    ws_c = workspace(kv.KV_OP_COMPACT, shape)
    ws_r = torch.zeros(kv.kv_recompact_workspace_size(max(cap, hkv * wl.n)), dtype=torch.uint8,
                       device=dev)
    budget = torch.tensor([total], dtype=torch.int64, device=dev)
    o = {"lb": torch.empty(B, L, dtype=torch.int32, device=dev),
         "hb": torch.empty(B, L, hkv, dtype=torch.int32, device=dev),
         "kept": torch.full((cap,), -7, dtype=torch.int32, device=dev),
         "cu": torch.zeros(B, L, hkv + 1, dtype=torch.int64, device=dev),
         "lens": torch.zeros(B, L, hkv, dtype=torch.int32, device=dev),
         "kf": torch.zeros(cap, wl.d, dtype=torch.bfloat16, device=dev),
         "vf": torch.zeros(cap, wl.d, dtype=torch.bfloat16, device=dev),
         "terms": torch.empty(B, L, hq, C, device=dev),
         "p": torch.empty(B, L, hkv, C, device=dev),
         "lb2": torch.empty(B, L, dtype=torch.int32, device=dev),
         "hb2": torch.empty(B, L, hkv, dtype=torch.int32, device=dev),
         "kept2": torch.full((cap,), -7, dtype=torch.int32, device=dev),
         "cu2": torch.zeros(B, L, hkv + 1, dtype=torch.int64, device=dev),
         "lens2": torch.zeros(B, L, hkv, dtype=torch.int32, device=dev),
         "kf2": torch.zeros(cap, wl.d, dtype=torch.bfloat16, device=dev),
         "vf2": torch.zeros(cap, wl.d, dtype=torch.bfloat16, device=dev)}

    def step(st):
        kv.kv_allocate_capped(shape, scores, budget, caps, 0, 1, o["lb"], o["hb"], ws_a, st)
        kv.kv_recompact(sh_old, scores[:, :L - 1], o["hb"][:, :L - 1], prev["kept"],
                        prev["cu"][:, :L - 1], prev["lens"][:, :L - 1], prev["kf"], prev["vf"],
                        2, None, o["kept"], o["cu"], o["lens"], o["kf"], o["vf"], ws_r, st)
        kv.kv_recompact(kv.KvShape.from_workload(wl, layers=1), scores[:, L - 1:],
                        o["hb"][:, L - 1:], None, None, None, inp["k"][:, L - 1:],
                        inp["v"][:, L - 1:], 2, o["cu"][0, L - 2, hkv:hkv + 1], o["kept"],
                        o["cu"][:, L - 1:], o["lens"][:, L - 1:], o["kf"], o["vf"], ws_r, st)
        kv.kv_window_terms(shape, kv.KV_TERMS_L2, inp["q_win"], inp["k"], o["terms"], ws_s, st)
        kv.kv_proj_score(shape, kv.KV_PROJ_LAPROX, inp["v"], w_oq, D, o["terms"], 0.0, o["p"],
                         ws_s, st)
        kv.kv_allocate(shape, o["p"], budget, 2, 0, 1, o["lb2"], o["hb2"], ws_a, st)
        kv.kv_compact(shape, inp["k"], inp["v"], o["p"], None, 1, 2, 0.0, o["hb2"], 2,
                      o["kept2"], o["cu2"], o["lens2"], o["kf2"], o["vf2"], cap, ws_c, st)

    st = torch.cuda.current_stream()
    step(st)
    torch.cuda.synchronize()
    eager = {k_: v_.clone() for k_, v_ in o.items()}
    for k_, v_ in o.items():     # back to the initial contents
        if k_.startswith("kept"):
            v_.fill_(-7)
        else:
            v_.zero_()
    gs = torch.cuda.Stream()
    gs.wait_stream(st)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=gs):
        step(gs)
    g.replay()
    torch.cuda.synchronize()
    for w_ in (ws_a, ws_s, ws_c, ws_r):
        assert kv.kv_check_device_status(w_) == 0
    for k_ in o:
        assert torch.equal(o[k_], eager[k_]), k_
