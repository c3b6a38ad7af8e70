"""Test helpers: drive the CUDA path through the C ABI, and the oracle on the same inputs."""
from __future__ import annotations

import math
from typing import Optional

import numpy as np
import torch

import kv_cache_eviction_gb300 as kv
import oracle as O

MODE = {"ada": kv.KV_SCORE_ADA, "lava": kv.KV_SCORE_LAVA, "critical": kv.KV_SCORE_CRITICAL}
GROUP = {"mean": kv.KV_GROUP_MEAN, "max": kv.KV_GROUP_MAX}


def workspace(op: int, shape, device="cuda") -> torch.Tensor:
    n = max(kv.kv_workspace_size(op, shape), 256)
    return torch.zeros(n, dtype=torch.uint8, device=device)


def capacity_rows(wl, B: int, L: int, budgets: torch.Tensor) -> int:
    if wl.budget_kind == "layer":
        return int(budgets.sum()) + B * L * wl.hkv * wl.reserve
    return int(budgets.sum()) + B * L * wl.hkv * wl.reserve


def run_score(wl, shape, inp, mode=None, group=None):
    mode = wl.mode if mode is None else mode
    group = wl.group if group is None else group
    B, L = shape.batch, shape.layers
    C = wl.n - wl.w
    dev = inp["k"].device
    scores = torch.empty(B, L, wl.hkv, C, dtype=torch.float32, device=dev)
    crit = torch.empty_like(scores) if mode == "critical" else None
    ws = workspace(kv.KV_OP_SCORE, shape)
    kv.kv_score(shape, MODE[mode], GROUP[group], inp["q_win"], inp["k"],
                inp["v"] if mode != "ada" else None, inp.get("w_o"), wl.model_dim, scores, crit, ws)
    assert kv.kv_check_device_status(ws) == 0
    return scores, crit


def run_allocate(wl, shape, scores, budgets, alpha=None):
    a, b = wl.alpha if alpha is None else alpha
    B, L = shape.batch, shape.layers
    dev = scores.device
    lb = torch.empty(B, L, dtype=torch.int32, device=dev)
    hb = torch.empty(B, L, wl.hkv, dtype=torch.int32, device=dev)
    ws = workspace(kv.KV_OP_ALLOCATE, shape)
    kv.kv_allocate(shape, scores, budgets.to(dev), 1 if wl.budget_kind == "total" else 0, a, b,
                   lb, hb, ws)
    assert kv.kv_check_device_status(ws) == 0
    return lb, hb


def run_compact(wl, shape, inp, scores, crit, hb, cap: int, reserve: Optional[int] = None):
    reserve = wl.reserve if reserve is None else reserve
    B, L = shape.batch, shape.layers
    dev = scores.device
    kept = torch.full((cap,), -7, dtype=torch.int32, device=dev)
    cu = torch.empty(B, L, wl.hkv + 1, dtype=torch.int64, device=dev)
    lens = torch.empty(B, L, wl.hkv, dtype=torch.int32, device=dev)
    kf = torch.zeros(cap, wl.d, dtype=wl.torch_dtype, device=dev)
    vf = torch.zeros(cap, wl.d, dtype=wl.torch_dtype, device=dev)
    ws = workspace(kv.KV_OP_COMPACT, shape)
    ca, cb = wl.crit_alpha
    kv.kv_compact(shape, inp["k"], inp["v"], scores, crit, ca, cb, wl.crit_eps, hb, reserve, kept,
                  cu, lens, kf, vf, cap, ws)
    assert kv.kv_check_device_status(ws) == 0
    return {"kept": kept, "cu": cu, "lens": lens, "kf": kf, "vf": vf}


def run_decode(wl, shape, q, kn, vn, flat, scale=None):
    dev = q.device
    scale = 1.0 / math.sqrt(wl.d) if scale is None else scale
    out = torch.empty_like(q)
    ws = workspace(kv.KV_OP_DECODE, shape)
    kv.flat_decode_attn(shape, q, kn, vn, flat["kf"], flat["vf"], flat["cu"], flat["lens"], scale,
                        out, ws)
    code = kv.kv_check_device_status(ws)
    return out, code


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def assert_scores_close(got: np.ndarray, ref: np.ndarray, rel=1e-4, abs_=1e-12, what="scores"):
    err = np.abs(got - ref)
    bad = err > rel * np.abs(ref) + abs_
    if bad.any():
        i = np.unravel_index(np.argmax(err / (rel * np.abs(ref) + abs_)), ref.shape)
        raise AssertionError("%s: %d of %d outside tolerance; worst at %s got %r ref %r" %
                             (what, int(bad.sum()), bad.size, i, got[i], ref[i]))


def oracle_kept_check(sg_oracle: np.ndarray, kept_gpu: np.ndarray, k: int, tie_rel=1e-5,
                      abs_floor=1e-12):
    """End-to-end per-head check: the GPU kept set may differ from the oracle's top-k only at
    near-ties (oracle score within tie_rel * tau of the oracle threshold tau)."""
    ref = O.topk_positions(sg_oracle, k)
    assert len(kept_gpu) == k
    assert np.all(np.diff(kept_gpu) > 0)
    diff = np.setxor1d(ref, kept_gpu)
    if diff.size == 0:
        return 0
    tau = np.sort(sg_oracle)[::-1][k - 1] if k > 0 else 0.0
    gap = np.abs(sg_oracle[diff] - tau)
    # scores below the 1e-12 absolute floor of the score tolerance count as ties too
    assert np.all(gap <= tie_rel * tau + abs_floor), (diff, sg_oracle[diff], tau)
    return diff.size
