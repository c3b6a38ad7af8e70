"""Plain fp64 CPU oracle of the "next" parts of the eviction method: LAVa's online layer-wise
prefill cascade, and selection from a cache that has already been compacted.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline``
/ ``--impl reference`` legs of ``bench.py`` may import this module; the library never does
and shares no code with it.  Every function follows the pages' definitions as loops and
single library primitives (a sort), with no blocking or fusion.

Pages (cited by title and section):

* "LAVa: Layer-wise KV Cache Eviction with Dynamic Budget Allocation" -- the online prefill
  and layer budget adjustment (after layer l is prefilled, the layers below it are
  compressed again with the same LAVa scores and budgets that shrink as more layers share
  the memory), uncertainty-based layer budgets, head-flattened layer eviction.

Readings taken where the pages are silent:

* Stage t (t = 1..L) starts when layer t-1 has been prefilled and scored.  The total
  budget (window rows included) is split over layers 0..t-1 exactly as the one-shot LAVa
  split does over all L layers -- R_t = total - t*w*Hkv selectable rows in proportion to the
  entropies e_l, floors plus largest remainders -- except that a layer can keep no more
  than it still holds: layer l < t-1 is capped at its selectable budget of stage t-1 and
  the new layer at Hkv*C.  While the prefilled layers cannot hold the whole budget (early
  stages of a large budget), each keeps everything it holds.  With caps that never bind,
  stage L reproduces the one-shot split.
* Each layer then keeps its head-flattened top B'_l (alpha = 0, the order (score desc, head
  asc, position asc)) chosen among the rows it still holds; the window rows stay.
"""
from __future__ import annotations

import math
from fractions import Fraction
from typing import List, Sequence

import numpy as np

from .kvevict_oracle import layer_entropy


def capped_split(e: Sequence[float], R: int, caps: Sequence[int]) -> np.ndarray:
    """R selectable rows shared by the layers in proportion to e_l, layer l at most caps[l].

    Layers whose proportional share exceeds their cap are fixed at the cap and the rest
    re-split; the others get floor(share) plus one each for the largest fractional parts
    (ties to the lower layer).  All-zero entropies split uniformly.  Exact rationals.  When
    R exceeds what the caps allow together, every layer keeps its cap.
    """
    L = len(e)
    if R < 0:
        raise ValueError("selectable total out of range")
    if R >= sum(int(c) for c in caps):
        return np.array([int(c) for c in caps], dtype=np.int64)
    ef = [Fraction(float(x)) for x in e]
    sel = [None] * L
    active = list(range(L))
    rem = Fraction(R)
    quota = {}
    while active:
        esum = sum(ef[l] for l in active)
        quota = {l: (rem * ef[l] / esum) if esum > 0 else rem / len(active) for l in active}
        over = [l for l in active if quota[l] > caps[l]]
        if not over:
            break
        for l in over:
            sel[l] = int(caps[l])
            rem -= int(caps[l])
        active = [l for l in active if l not in over]
    fl = {l: math.floor(quota[l]) for l in active}
    for l in active:
        sel[l] = fl[l]
    left = int(rem) - sum(fl.values())
    for l in sorted(active, key=lambda x: (-(quota[x] - fl[x]), x))[:left]:
        sel[l] += 1
    return np.array(sel, dtype=np.int64)


def layer_top_from_held(s: np.ndarray, held: List[np.ndarray], Bp: int) -> List[np.ndarray]:
    """The layer-wide top B' (score desc, head asc, position asc) among the candidate
    positions each head still holds; returns the chosen positions per head, ascending."""
    hkv = s.shape[0]
    vals, heads, pos = [], [], []
    for g in range(hkv):
        vals.append(s[g][held[g]])
        heads.append(np.full(len(held[g]), g))
        pos.append(held[g])
    vals = np.concatenate(vals) if vals else np.zeros(0)
    heads = np.concatenate(heads).astype(np.int64)
    pos = np.concatenate(pos).astype(np.int64)
    if Bp > len(vals):
        raise ValueError("budget larger than the rows held")
    order = np.lexsort((pos, heads, -vals))[:Bp]
    return [np.sort(pos[order][heads[order] == g]) for g in range(hkv)]


def lava_cascade(S: Sequence[np.ndarray], total: int, w: int, n: int) -> List[dict]:
    """LAVa's online layer-wise prefill with budget adjustment, stage by stage.

    S[l] [Hkv, C] are the LAVa scores of layer l (window mean, pooled, group max, times
    max_k ||V[k]||_1), total the budget of the whole sequence with every window included.
    Returns one dict per stage t = 1..L:
      layer_budget [t]      B_l including the w*Hkv window rows (sum = total, or less while
                            the prefilled layers cannot hold that much)
      head_budget  [t][Hkv] kept rows per head, window included
      kept         [t][Hkv] kept positions per head, ascending, window last
      rows_before           rows held while layer t-1 has just been prefilled (the
                            earlier layers' kept rows plus the new layer's n*Hkv)
      rows_after            rows held once the stage's compression is done
      caps_bound            whether some layer's cap held it below its proportional share
    """
    L = len(S)
    hkv, C = S[0].shape
    e = [layer_entropy(np.asarray(S[l], dtype=np.float64), n) for l in range(L)]
    held: List[List[np.ndarray]] = []
    prev_sel: List[int] = []
    stages = []
    for t in range(1, L + 1):
        R = total - t * w * hkv
        caps = [min(hkv * C, int(prev_sel[l])) for l in range(t - 1)] + [hkv * C]
        sel = capped_split(e[:t], R, caps)
        uncapped = capped_split(e[:t], R, [hkv * C] * t)
        rows_before = sum(int(x) + w * hkv for x in prev_sel) + n * hkv
        new_held = []
        for l in range(t):
            cand = held[l] if l < t - 1 else [np.arange(C)] * hkv
            new_held.append(layer_top_from_held(np.asarray(S[l], dtype=np.float64), cand,
                                                int(sel[l])))
        held = new_held
        prev_sel = [int(x) for x in sel]
        stages.append({
            "layer_budget": sel + w * hkv,
            "head_budget": np.array([[len(held[l][g]) + w for g in range(hkv)]
                                     for l in range(t)], dtype=np.int64),
            "kept": [[np.concatenate([held[l][g], np.arange(C, n)]).astype(np.int64)
                      for g in range(hkv)] for l in range(t)],
            "rows_before": rows_before,
            "rows_after": int(sel.sum()) + t * w * hkv,
            "caps_bound": bool(np.any(sel != uncapped)),
        })
    return stages
