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
@pytest.mark.parametrize("path", [None, "split", "rows"])
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
