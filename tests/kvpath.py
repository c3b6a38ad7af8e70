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


def oracle_crit_kept_check(s_ref: np.ndarray, c_ref: np.ndarray, s_gpu: np.ndarray,
                           kept_gpu: np.ndarray, k: int, a: int, b: int, eps: float,
                           tie_rel=1e-5, abs_floor=1e-12):
    """End-to-end check of one head's CriticalKV two-stage selection.

    The GPU's stage-1 set is recovered from its kept rows: the floor(a/b * k) of them that
    rank highest by the GPU's own float32 scores (stage 1 is the top of every candidate by
    that order, so it is the top of the kept rows too).  Then
      - stage 1 may differ from the oracle's top by s only at s near-ties (oracle_kept_check);
      - the rest of the kept rows must be the top k - k1 of the candidates outside the GPU's
        stage 1, ranked by the oracle's kappa = (s + eps) * c, up to kappa near-ties.
    Returns the number of positions that differ from the oracle's own two-stage result."""
    assert len(kept_gpu) == k
    assert np.all(np.diff(kept_gpu) > 0)
    k1 = (a * k) // b
    order = np.lexsort((kept_gpu, -s_gpu[kept_gpu].astype(np.float64)))
    st1 = np.sort(kept_gpu[order[:k1]])
    oracle_kept_check(s_ref, st1, k1, tie_rel, abs_floor)
    st2 = np.setdiff1d(kept_gpu, st1)
    rest = np.setdiff1d(np.arange(len(s_ref)), st1)
    kappa = (s_ref + eps) * c_ref
    k2 = k - k1
    ref2 = rest[np.lexsort((rest, -kappa[rest]))[:k2]]
    diff = np.setxor1d(ref2, st2)
    if diff.size:
        tau = np.sort(kappa[rest])[::-1][k2 - 1]
        gap = np.abs(kappa[diff] - tau)
        assert np.all(gap <= tie_rel * tau + abs_floor), (diff, kappa[diff], tau)
    full = O.critical_positions(s_ref, c_ref, k, a, b, eps)
    return int(np.setxor1d(full, kept_gpu).size)


def assert_decode_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = "decode",
                        atol: float = None) -> float:
    """The decode bar against the fp64 oracle; returns the plain max-abs error.

    bf16: 1e-2 max-abs, applied to the float32-accumulated result.  The ABI stores the output
    in bf16, whose rounding adds up to half an ulp (at most 2^-8 |ref|).  Below |ref| = 4 that
    half ulp is at most 2^-7 < 1e-2, so there the plain bar |got - ref| <= 1e-2 is asserted as
    it stands; at |ref| >= 4 (where no bf16 value could meet a plain 1e-2) the half ulp is
    added to it.  float32 (stored as computed): 1e-4 max-abs.
    """
    err = np.abs(got - ref)
    if dtype == "bf16":
        a = 1e-2 if atol is None else atol
        small = np.abs(ref) < 4.0
        ok = np.where(small, err <= a, err <= a + 2.0 ** -8 * np.abs(ref))
    else:
        a = 1e-4 if atol is None else atol
        ok = err <= a
    plain = float(err.max()) if err.size else 0.0
    small_err = float(err[np.abs(ref) < 4.0].max()) if (np.abs(ref) < 4.0).any() else 0.0
    print("%s: plain max-abs err %.3e (%.3e where |ref| < 4), max |ref| %.3g" %
          (what, plain, small_err, float(np.abs(ref).max()) if ref.size else 0.0))
    if not ok.all():
        i = np.unravel_index(np.argmax(np.where(ok, 0.0, err)), err.shape)
        raise AssertionError("%s: %d outside the decode bar; worst at %s got %r ref %r" %
                             (what, int((~ok).sum()), i, got[i], ref[i]))
    return plain
