"""flat_decode_attn_noalloc: the decode step for callers that cannot allocate device memory.

Such callers (a serving loop with a fixed memory plan, a plugin handed only its buffers, work
issued during stream capture) get the decode without passing a workspace; the library uses a
fixed scratch array compiled into it.  This file runs last (pytest collects it after the others)
so that a failure here never hides the other tests' results.  It must pass alone in a fresh
process and after every other test in the same process.
"""
import ctypes
import math
import os

import pytest
import torch

import kv_cache_eviction_gb300 as kv
from kv_cache_eviction_gb300 import workloads as W
from tests.kvpath import capacity_rows, run_allocate, run_compact, run_decode, run_score

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_eviction_gb300 import _build
    _build.build()
    kv.lib()


@pytest.fixture(params=["default", "split", "heads", "rows", "parts"])
def decode_path(request):
    """Each decode kernel on the fixed scratch: the default choice, then the one-launch split
    (tickets and partials in the scratch), one CTA per KV head (only the error word there), the
    row-balanced split (chunk map, work counter and partials there) and the heads in parts
    (per-head tickets, a done counter and partials there)."""
    old = os.environ.get("KVEVICT_DECODE_PATH")
    if request.param == "default":
        os.environ.pop("KVEVICT_DECODE_PATH", None)
    else:
        os.environ["KVEVICT_DECODE_PATH"] = request.param
    yield request.param
    if old is None:
        os.environ.pop("KVEVICT_DECODE_PATH", None)
    else:
        os.environ["KVEVICT_DECODE_PATH"] = old


def _flat_copy(flat):
    return {k: v.clone() for k, v in flat.items()}


def test_noalloc_decode_matches_workspace_decode_twice(decode_path):
    """Two decode steps in a row through both entry points on copies of one flat cache.  Both
    run the same kernels on the same inputs, so outputs, appended rows and lengths must be
    identical bit for bit; the second step also sees whatever the first left in the shared
    scratch."""
    wl = W.Workload(name="noalloc", batch=2, layers=3, hq=32, hkv=8, d=128, n=3000, w=32, pool=7,
                    dtype="bf16", temp=(0.5, 16.0), head_budget_tokens=600, reserve=4, seed=99)
    B, L = wl.batch, wl.layers
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    scores, _ = run_score(wl, shape, inp)
    budgets = wl.budgets()
    _, hb = run_allocate(wl, shape, scores, budgets)
    flat = run_compact(wl, shape, inp, scores, None, hb, capacity_rows(wl, B, L, budgets))
    flat_a, flat_b = _flat_copy(flat), _flat_copy(flat)
    scale = 1.0 / math.sqrt(wl.d)
    for step in range(2):
        dec = W.make_decode_batch(wl, step, inp["tau"], device="cuda")
        out_a, code = run_decode(wl, shape, dec["q"], dec["k_new"], dec["v_new"], flat_a)
        assert code == 0
        out_b = torch.full_like(dec["q"], float("nan"))
        kv.flat_decode_attn_noalloc(shape, dec["q"], dec["k_new"], dec["v_new"], flat_b["kf"],
                                    flat_b["vf"], flat_b["cu"], flat_b["lens"], scale, out_b)
        torch.cuda.synchronize()
        assert torch.equal(out_a, out_b), (step, (out_a.float() - out_b.float()).abs().max())
        assert torch.equal(flat_a["lens"], flat_b["lens"])
        assert torch.equal(flat_a["kf"], flat_b["kf"]) and torch.equal(flat_a["vf"], flat_b["vf"])


def test_noalloc_rejects_decodes_larger_than_its_scratch():
    shape = kv.KvShape.of(batch=64, layers=32, hq=32, hkv=8, d=128, n=65536, w=32, pool=7,
                          dtype="bf16")
    assert kv.kv_workspace_size(kv.KV_OP_DECODE, shape) > (16 << 20)
    p = ctypes.c_void_p(1 << 20)
    st = kv.lib().flat_decode_attn_noalloc(ctypes.byref(shape), p, None, None, p, p, p, p, 1 << 30,
                                           0.1, p, None)
    assert st == kv.KV_ERR_WORKSPACE
