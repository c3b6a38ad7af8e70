"""The tcgen05 window-scoring path (bf16, d = 128, G*w = 128) against the oracle, and the
CUDA-core path on the same inputs.  Shapes cover ragged n, every supported w, several
units per launch (the P1/P2 interleave and the cross-CTA LSE publication) and LAVa."""
import os
import zlib

import numpy as np
import pytest
import torch

import kv_cache_eviction_gb300 as kv
from kv_cache_eviction_gb300 import workloads as W
from tests.kvpath import assert_scores_close, np64, run_score
from tests.test_gpu_parity import oracle_scores

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cache_eviction_gb300 import _build
    _build.build()
    kv.lib()


def score_with(path, wl, shape, inp):
    old = os.environ.get("KVEVICT_SCORE_PATH")
    os.environ["KVEVICT_SCORE_PATH"] = path
    try:
        n0 = kv.kv_kernel_launches()
        s, _ = run_score(wl, shape, inp)
        torch.cuda.synchronize()
        return s.cpu().numpy(), kv.kv_kernel_launches() - n0
    finally:
        if old is None:
            del os.environ["KVEVICT_SCORE_PATH"]
        else:
            os.environ["KVEVICT_SCORE_PATH"] = old


CASES = [
    # name, hq, hkv, w, n, batch, layers, mode, group, pool
    ("w32_ragged", 32, 8, 32, 5000 + 13, 1, 1, "ada", "mean", 7),
    ("w16_g8", 64, 8, 16, 2500, 1, 1, "ada", "mean", 7),
    ("w64_g2", 16, 8, 64, 3000, 1, 2, "ada", "max", 5),
    ("short_n", 8, 2, 32, 130, 1, 1, "ada", "mean", 7),
    ("many_units", 8, 2, 32, 1000, 3, 4, "ada", "mean", 7),
    ("lava_units", 32, 8, 32, 4100, 1, 3, "lava", "max", 7),
    ("pool1", 8, 2, 32, 700, 1, 2, "ada", "mean", 1),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_tc_scores_match_oracle(case):
    name, hq, hkv, w, n, B, L, mode, group, pool = case
    wl = W.Workload(name=name, batch=B, layers=L, hq=hq, hkv=hkv, d=128, n=n, w=w, pool=pool,
                    dtype="bf16", temp=(0.5, 16.0), v_lognormal=0.5 if mode == "lava" else 0.0,
                    mode=mode, group=group, head_budget_tokens=8, seed=zlib.crc32(name.encode()) & 0xFFFF)
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    s_tc, launches_tc = score_with("tc", wl, shape, inp)
    s_simt, launches_simt = score_with("simt", wl, shape, inp)
    # the tensor-core path is one main kernel (+ the V-bar pass, + the halo fix-up)
    assert launches_tc < launches_simt
    for b in range(B):
        for l in range(L):
            q = np64(inp["q_win"][b, l])
            k = np64(inp["k"][b, l])
            v = np64(inp["v"][b, l])
            ref, _ = oracle_scores(wl, q, k, v)
            assert_scores_close(s_tc[b, l].astype(np.float64), ref, what="tc b%d l%d" % (b, l))
            assert_scores_close(s_simt[b, l].astype(np.float64), ref,
                                what="simt b%d l%d" % (b, l))


CRIT_CASES = [
    # name, n, D, batch, layers, hkv: ragged key tails, D not a multiple of the 128-column
    # tile, several (layer, KV head) output blocks
    ("crit_ragged", 1000 + 7, 1000, 2, 2, 2),
    ("crit_d4096", 600, 4096, 1, 1, 8),
    ("crit_tiny_c", 40, 136, 1, 3, 2),
]


@pytest.mark.parametrize("case", CRIT_CASES, ids=[c[0] for c in CRIT_CASES])
def test_crit_norm_tc_matches_oracle(case):
    """||(V W_O)_j||_1 on the tensor cores (one MN-major W_O operand per (layer, KV head))
    against the oracle's fp64 product, and the CUDA-core kernel on the same inputs."""
    import oracle as O
    name, n, D, B, L, hkv = case
    wl = W.Workload(name=name, batch=B, layers=L, hq=4 * hkv, hkv=hkv, d=128, n=n, w=32, pool=7,
                    dtype="bf16", temp=(0.5, 16.0), mode="critical", head_budget_frac=0.4,
                    model_dim=D, seed=zlib.crc32(name.encode()) & 0xFFFF)
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    crits = {}
    for path in ("tc", "simt"):
        old = os.environ.get("KVEVICT_SCORE_PATH")
        os.environ["KVEVICT_SCORE_PATH"] = path
        try:
            _, c = run_score(wl, shape, inp)
            crits[path] = c.cpu().numpy()
        finally:
            if old is None:
                del os.environ["KVEVICT_SCORE_PATH"]
            else:
                os.environ["KVEVICT_SCORE_PATH"] = old
    C = n - wl.w
    for b in range(B):
        for l in range(L):
            ref = O.critical_row_norm(np64(inp["v"][b, l]), np64(inp["w_o"][l]), C)
            for path, c in crits.items():
                assert_scores_close(c[b, l].astype(np.float64), ref,
                                    what="crit %s b%d l%d" % (path, b, l))


def test_crit_norm_entry_equals_score_output():
    """kv_crit_norm alone writes exactly what kv_score writes to crit_norm in CriticalKV
    mode (the same kernel), and matches the oracle."""
    import oracle as O
    wl = W.Workload(name="critnorm", batch=1, layers=2, hq=8, hkv=2, d=128, n=1000, w=32, pool=7,
                    dtype="bf16", temp=(0.5, 16.0), mode="critical", head_budget_frac=0.4,
                    model_dim=520, seed=21)
    shape = kv.KvShape.from_workload(wl)
    inp = W.make_batch(wl, device="cuda")
    _, c_score = run_score(wl, shape, inp)
    c_alone = torch.full_like(c_score, float("nan"))
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    kv.kv_crit_norm(shape, inp["v"], inp["w_o"], wl.model_dim, c_alone, ws)
    assert kv.kv_check_device_status(ws) == 0
    assert torch.equal(c_alone, c_score)
    C = wl.n - wl.w
    for l in range(wl.layers):
        ref = O.critical_row_norm(np64(inp["v"][0, l]), np64(inp["w_o"][l]), C)
        assert_scores_close(c_alone[0, l].double().cpu().numpy(), ref, what="crit l%d" % l)
