"""The C ABI without a GPU: the library builds, loads, exports every declared symbol, and
rejects invalid arguments on the host before anything is enqueued."""
import ctypes
import os
import re

import pytest

import kv_cache_eviction_gb300 as kv
from kv_cache_eviction_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    _build.build()
    return kv.lib()


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"KV_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)
    return names


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert {"kv_score", "kv_allocate", "kv_compact", "flat_decode_attn", "kv_workspace_size",
            "kv_check_device_status", "kv_status_string"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code in range(7):
        s = kv.kv_status_string(code)
        assert s and s != "unknown status"
    assert kv.kv_status_string(99) == "unknown status"


def shape(**kw):
    base = dict(batch=1, layers=2, hq=32, hkv=8, d=128, n=4096, w=32, pool=7, dtype="bf16")
    base.update(kw)
    return kv.KvShape.of(**base)


def test_workspace_sizes(L):
    s = shape()
    for op in range(4):
        assert kv.kv_workspace_size(op, s) >= 256
    assert kv.kv_workspace_size(9, s) == 0
    assert kv.kv_workspace_size(0, shape(d=100)) == 0      # d not a multiple of 8
    assert kv.kv_workspace_size(0, shape(w=5000)) == 0     # window longer than the prefix
    assert kv.kv_workspace_size(0, shape(pool=6)) == 0     # even pool width
    assert kv.kv_workspace_size(0, shape(hq=30)) == 0      # Hq not a multiple of Hkv


@pytest.mark.parametrize("bad", [dict(d=100), dict(w=5000), dict(pool=4), dict(hq=12, hkv=8),
                                 dict(dtype=7), dict(batch=-1)])
def test_invalid_shapes_rejected_on_host(L, bad):
    s = shape(**bad)
    buf = ctypes.c_void_p(0x1000)
    assert L.kv_score(ctypes.byref(s), 0, 0, buf, buf, None, None, 0, buf, None, buf, 1 << 20,
                      None) == kv.KV_ERR_INVALID_ARG
    assert L.kv_allocate(ctypes.byref(s), buf, buf, 0, 1, 5, buf, buf, buf, 1 << 20,
                         None) == kv.KV_ERR_INVALID_ARG
    assert L.kv_compact(ctypes.byref(s), buf, buf, buf, None, 1, 2, 0.0, buf, 0, buf, buf, buf,
                        buf, buf, 1 << 20, buf, 1 << 20, None) == kv.KV_ERR_INVALID_ARG
    assert L.flat_decode_attn(ctypes.byref(s), buf, None, None, buf, buf, buf, buf, 1 << 20, 0.1,
                              buf, buf, 1 << 20, None) == kv.KV_ERR_INVALID_ARG


def test_invalid_parameters_rejected_on_host(L):
    s = shape()
    p = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1004)
    assert L.kv_score(None, 0, 0, p, p, None, None, 0, p, None, p, 1 << 20, None) == 1
    assert L.kv_score(ctypes.byref(s), 5, 0, p, p, None, None, 0, p, None, p, 1 << 20, None) == 1
    assert L.kv_score(ctypes.byref(s), 0, 3, p, p, None, None, 0, p, None, p, 1 << 20, None) == 1
    assert L.kv_score(ctypes.byref(s), 0, 0, p, p, None, None, 0, p, None, None, 0, None) == 1
    assert L.kv_score(ctypes.byref(s), 0, 0, odd, p, None, None, 0, p, None, p, 1 << 30, None) == 1
    # LAVa and CriticalKV need v; CriticalKV needs w_o, crit_norm and model_dim % 8 == 0
    assert L.kv_score(ctypes.byref(s), 1, 1, p, p, None, None, 0, p, None, p, 1 << 30, None) == 1
    assert L.kv_score(ctypes.byref(s), 2, 0, p, p, p, None, 4096, p, p, p, 1 << 30, None) == 1
    assert L.kv_score(ctypes.byref(s), 2, 0, p, p, p, p, 4090, p, p, p, 1 << 30, None) == 1
    # alpha must be a fraction in [0, 1] with a denominator <= 65536
    for a, b in [(1, 0), (3, 2), (1, 1 << 20)]:
        assert L.kv_allocate(ctypes.byref(s), p, p, 0, a, b, p, p, p, 1 << 30, None) == 1
    assert L.kv_allocate(ctypes.byref(s), p, p, 3, 1, 5, p, p, p, 1 << 30, None) == 1
    # k_new without v_new
    assert L.flat_decode_attn(ctypes.byref(s), p, p, None, p, p, p, p, 1 << 20, 0.1, p, p,
                              1 << 30, None) == 1
    assert L.flat_decode_attn(ctypes.byref(s), p, None, None, p, p, p, p, 1 << 20,
                              ctypes.c_float(float("nan")), p, p, 1 << 30, None) == 1
    assert L.flat_decode_attn(ctypes.byref(s), p, None, None, p, p, p, p, -1, 0.1, p, p,
                              1 << 30, None) == 1
    # negative reserve, and a flat buffer that cannot even hold the windows
    assert L.kv_compact(ctypes.byref(s), p, p, p, None, 1, 2, 0.0, p, -1, p, p, p, p, p, 1 << 20,
                        p, 1 << 30, None) == 1
    assert L.kv_compact(ctypes.byref(s), p, p, p, None, 1, 2, 0.0, p, 0, p, p, p, p, p, 10, p,
                        1 << 30, None) == kv.KV_ERR_CAPACITY
    # CriticalKV stage-1 fraction and eps
    assert L.kv_compact(ctypes.byref(s), p, p, p, p, 3, 2, 0.0, p, 0, p, p, p, p, p, 1 << 20, p,
                        1 << 30, None) == 1
    assert L.kv_compact(ctypes.byref(s), p, p, p, p, 1, 2, ctypes.c_float(-1.0), p, 0, p, p, p, p,
                        p, 1 << 20, p, 1 << 30, None) == 1


def test_short_workspace_rejected_on_host(L):
    """A workspace one byte short of kv_workspace_size is refused before anything is
    enqueued (the decode plan includes the split kernel's counters and tickets)."""
    s = shape()
    p = ctypes.c_void_p(0x1000)
    n = [kv.kv_workspace_size(op, s) for op in range(4)]
    assert L.kv_score(ctypes.byref(s), 0, 0, p, p, None, None, 0, p, None, p, n[0] - 1,
                      None) == kv.KV_ERR_WORKSPACE
    assert L.kv_allocate(ctypes.byref(s), p, p, 0, 1, 5, p, p, p, n[1] - 1,
                         None) == kv.KV_ERR_WORKSPACE
    # (the compaction size covers CriticalKV's stage-1 flags: pass a norm array)
    assert L.kv_compact(ctypes.byref(s), p, p, p, p, 1, 2, 0.0, p, 0, p, p, p, p, p, 1 << 20,
                        p, n[2] - 1, None) == kv.KV_ERR_WORKSPACE
    assert L.flat_decode_attn(ctypes.byref(s), p, None, None, p, p, p, p, 1 << 20, 0.1, p, p,
                              n[3] - 1, None) == kv.KV_ERR_WORKSPACE
    # the decode plan grows with the heads: one ticket per KV head at least
    big = shape(batch=4 * s.batch)
    assert kv.kv_workspace_size(3, big) >= n[3] + 3 * s.batch * s.layers * s.hkv * 4


def test_empty_batch_is_a_no_op(L):
    s = shape(batch=0)
    p = ctypes.c_void_p(0x1000)
    assert L.kv_score(ctypes.byref(s), 0, 0, None, None, None, None, 0, None, None, p, 256,
                      None) == kv.KV_OK
    assert L.kv_allocate(ctypes.byref(s), None, None, 0, 1, 5, None, None, p, 256, None) == 0
    assert L.kv_compact(ctypes.byref(s), None, None, None, None, 1, 2, 0.0, None, 0, None, None,
                        None, None, None, 0, p, 256, None) == 0
    assert L.flat_decode_attn(ctypes.byref(s), None, None, None, None, None, None, None, 0, 0.1,
                              None, p, 256, None) == 0


def test_binding_refuses_host_tensors(L):
    import torch
    s = shape()
    t = torch.zeros(16)
    with pytest.raises(ValueError):
        kv.kv_score(s, 0, 0, t, t, None, None, 0, t, None, t)


def test_next_calls_reject_invalid_arguments_on_host(L):
    """The calls of the cascade, the per-query-head scores and the presets refuse bad
    arguments before anything is enqueued (no GPU is touched here)."""
    s = shape()
    p = ctypes.c_void_p(0x1000)
    odd = ctypes.c_void_p(0x1004)
    big = 1 << 30
    # kv_allocate_capped: caps required, alpha a fraction
    assert L.kv_allocate_capped(ctypes.byref(s), p, p, None, 0, 1, p, p, p, big, None) == 1
    assert L.kv_allocate_capped(ctypes.byref(s), p, p, p, 2, 1, p, p, p, big, None) == 1
    assert L.kv_allocate_capped(ctypes.byref(s), p, p, p, 0, 1, p, p, p,
                                kv.kv_workspace_size(1, s) - 1, None) == kv.KV_ERR_WORKSPACE
    # kv_recompact: the source is a flat cache (all three tables) or the K/V (none); the
    # output is not the source; row tables and rows aligned; workspace large enough
    vout = ctypes.c_void_p(0x3000)
    args = lambda kept, cu, lens, sk, out, ws_bytes: (
        ctypes.byref(s), p, p, kept, cu, lens, sk, p, 1 << 20, 0, None, p, p, p, out, vout,
        1 << 20, p, ws_bytes, None)
    assert L.kv_recompact(*args(p, None, p, p, ctypes.c_void_p(0x2000), big)) == 1
    assert L.kv_recompact(*args(p, p, p, p, p, big)) == 1                    # k_flat is src_k
    assert L.kv_recompact(*args(p, p, p, odd, ctypes.c_void_p(0x2000), big)) == 1
    assert L.kv_recompact(*args(p, p, p, p, ctypes.c_void_p(0x2000),
                                kv.kv_recompact_workspace_size(1 << 20) - 1)) == 3
    assert kv.kv_recompact_workspace_size(-1) == 0
    # kv_window_terms / kv_proj_score: kind, eps, model_dim
    assert L.kv_window_terms(ctypes.byref(s), 2, p, p, p, p, big, None) == 1
    assert L.kv_window_terms(ctypes.byref(s), 0, odd, p, p, p, big, None) == 1
    assert L.kv_proj_score(ctypes.byref(s), 2, p, p, 4096, p, 0.0, p, p, big, None) == 1
    assert L.kv_proj_score(ctypes.byref(s), 0, p, p, 4090, p, 0.0, p, p, big, None) == 1
    assert L.kv_proj_score(ctypes.byref(s), 0, p, p, 4096, p, ctypes.c_float(-1.0), p, p, big,
                           None) == 1
    assert L.kv_proj_score(ctypes.byref(shape(dtype="f32", d=64)), 0, p, p, 4096, p, 0.0, p, p,
                           big, None) == kv.KV_ERR_UNSUPPORTED
    # kv_compact_kappa / kv_compact_streaming: kappa required, alpha a fraction, sinks >= 0
    assert L.kv_compact_kappa(ctypes.byref(s), p, p, p, None, 1, 2, p, 0, p, p, p, p, p, 1 << 20,
                              p, big, None) == 1
    assert L.kv_compact_kappa(ctypes.byref(s), p, p, p, p, 3, 2, p, 0, p, p, p, p, p, 1 << 20,
                              p, big, None) == 1
    assert L.kv_compact_streaming(ctypes.byref(s), p, p, -1, p, 0, p, p, p, p, p, 1 << 20, p,
                                  big, None) == 1
    assert L.kv_compact_streaming(ctypes.byref(s), p, p, 4, p, 0, p, p, p, p, p, 10, p, big,
                                  None) == kv.KV_ERR_CAPACITY
    # the model-wide allocation needs L * Hkv <= 256
    wide = shape(layers=64)
    assert L.kv_allocate(ctypes.byref(wide), p, p, 2, 0, 1, p, p, p, big,
                         None) == kv.KV_ERR_UNSUPPORTED
    # kv_crit_norm: model_dim a multiple of 8
    assert L.kv_crit_norm(ctypes.byref(s), p, p, 4090, p, p, big, None) == 1
