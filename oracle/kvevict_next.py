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

* "CriticalKV: Optimizing KV Cache Eviction from an Output Perturbation Perspective" -- key
  designs: the bound weighs entry i by ||(V W^O)_{i,:}||_1 per head, and the two-stage
  greedy selection (top alpha*b by A, then the rest by (A_i + eps) * ||(V W^O)_i||_1);
  "Ada-KV" notes, efficiency section, GQA: the mean over a group as the criterion.
* "Ada-KV" arXiv page, Parameters: the sliding-window baseline (StreamingLLM) keeps 4 sink
  tokens and the most recent window's cache.
* "CriticalKV" notes, limitations: how to re-select when new entries join the cache during
  decoding (streaming, chunked prefill) is left open.
* "Reformulating KV cache eviction for long-context LLM inference" (LaProx) -- Eqs. 2-4
  (the output is the sum of the heads' contributions A^(h) V^(h) W_O^(h)) and Algorithm 1:
  p[i] = ||A[:, i]||_2 * ||H[i, :]||_2 with A the window's attention rows and H = V W_O,
  the last w entries always kept, then one TopK over the budget B_total.

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
* StreamingLLM as a budget preset: head g keeps its first min(sinks, B_g) positions and the
  B_g - that many most recent candidates before the window (the window itself always
  stays): the recent window grows into the candidates to fill the same budget an adaptive
  head would get.
* Re-eviction during decoding: the rows appended by decode steps carry no prefill score;
  they are the cache's newest tokens and stay, like the window.  To return to a smaller
  budget, each head keeps its top prefill rows by the prefill scores among those it still
  holds.
* GQA-exact CriticalKV: W^O is split per query head (the [d, D] block of head q's rows of
  the model's output projection), so KV head g's rows meet G different blocks.  The
  composite score of query head q is (A_q[i] + eps) * ||(V_g W^O_q)_i||_1 with A_q that
  head's pooled window mean; the KV head's score is their mean over the group (Ada-KV's
  GQA criterion).  Stage 1 stays the Ada-KV score (group mean of A_q).  With one W^O block
  shared by the group this is exactly the per-KV-head form (s + eps) * ||(V W^O)_i||_1.
* LaProx under GQA: the output is a sum over query heads, so KV head g's entry i carries
  sum_{q in g} ||A_q[:, i]||_2 * ||(V_g W^O_q)_i||_2 (the bound of the Frobenius norm of
  the entry's contribution to the window's outputs; one term for MHA, as on the page).
  ||A_q[:, i]||_2 is over the w window rows with no pooling (Algorithm 1 prints none).
  B_total is the whole model's budget with every window included; TopK runs over every
  candidate of every layer and KV head at once (the page's model-wide selection), ties by
  (layer, head, position) ascending.
"""
from __future__ import annotations

import math
from fractions import Fraction
from typing import List, Sequence

import numpy as np

from .kvevict_oracle import global_topk_counts, layer_entropy, max_pool, window_attention


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


# ----------------------------------------------------------------------------
# Per-query-head terms: CriticalKV with one W^O block per query head, and LaProx.
# ----------------------------------------------------------------------------

def window_head_terms(q_win: np.ndarray, k: np.ndarray, w: int, pool: int, kind: str,
                      scale=None) -> np.ndarray:
    """The window term of every query head for every candidate j < C, before any group
    reduction.  q_win [Hq, w, d], k [Hkv, n, d] -> [Hq, C].

    ``mean_pool``: max_pool(window mean of P_q) -- Ada-KV's per-head score (Algorithm 2);
    ``l2``:        sqrt(sum_t P_q[t, j]^2) -- LaProx's ||A[:, j]||_2, no pooling.
    P is the causal window attention over all n keys (as for the Ada-KV scores).
    """
    n, d = k.shape[1], k.shape[2]
    C = n - w
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    P = window_attention(q_win, k, scale)
    if kind == "mean_pool":
        return max_pool(P[:, :, :C].mean(axis=1), pool) if C > 0 else np.zeros((len(P), 0))
    if kind == "l2":
        return np.sqrt((P[:, :, :C] ** 2).sum(axis=1))
    raise ValueError(kind)


def head_proj_norm(v: np.ndarray, w_o_q: np.ndarray, C: int, p: int) -> np.ndarray:
    """||(V_g W^O_q)_j||_p for every query head q (KV head g = q // G) and j < C.

    v [Hkv, n, d], w_o_q [Hq, d, D] -> [Hq, C]."""
    hkv = v.shape[0]
    hq = w_o_q.shape[0]
    G = hq // hkv
    out = np.empty((hq, C))
    for q in range(hq):
        proj = v[q // G, :C].astype(np.float64) @ w_o_q[q].astype(np.float64)
        if p == 1:
            out[q] = np.abs(proj).sum(axis=1)
        elif p == 2:
            out[q] = np.sqrt((proj ** 2).sum(axis=1))
        else:
            raise ValueError(p)
    return out


def gqa_critical_kappa(terms: np.ndarray, v: np.ndarray, w_o_q: np.ndarray, eps: float
                       ) -> np.ndarray:
    """CriticalKV's stage-2 key with one W^O block per query head, group mean:
    kappa[g, j] = (1/G) sum_{q in g} (A_q[j] + eps) * ||(V_g W^O_q)_j||_1.
    terms [Hq, C] (window_head_terms 'mean_pool') -> [Hkv, C]."""
    hq, C = terms.shape
    hkv = v.shape[0]
    G = hq // hkv
    c = head_proj_norm(v, w_o_q, C, 1)
    kap = np.zeros((hkv, C))
    for q in range(hq):
        kap[q // G] += (terms[q] + eps) * c[q]
    return kap / G


def laprox_score(terms: np.ndarray, v: np.ndarray, w_o_q: np.ndarray) -> np.ndarray:
    """LaProx's entry score, per KV head: p[g, j] = sum_{q in g} ||A_q[:, j]||_2 *
    ||(V_g W^O_q)_j||_2.  terms [Hq, C] (window_head_terms 'l2') -> [Hkv, C]."""
    hq, C = terms.shape
    hkv = v.shape[0]
    G = hq // hkv
    h = head_proj_norm(v, w_o_q, C, 2)
    p = np.zeros((hkv, C))
    for q in range(hq):
        p[q // G] += terms[q] * h[q]
    return p


def laprox_head_budgets(P: Sequence[np.ndarray], total: int, w: int) -> np.ndarray:
    """LaProx's model-wide TopK: the top (total - L*w*Hkv) candidates over every layer's
    every KV head at once (order: score desc, then layer, head, position ascending), counted
    per (layer, head).  P[l] [Hkv, C].  Returns the kept rows per (layer, head) [L, Hkv],
    window included."""
    L = len(P)
    hkv, C = P[0].shape
    Bp = total - L * w * hkv
    if Bp < 0 or Bp > L * hkv * C:
        raise ValueError("total budget out of range")
    f = global_topk_counts(np.concatenate([np.asarray(x, dtype=np.float64) for x in P]), Bp)
    return f.reshape(L, hkv) + w


def critical_positions_kappa(sg: np.ndarray, kg: np.ndarray, k: int, a: int, b: int
                             ) -> np.ndarray:
    """CriticalKV's two-stage selection with the stage-2 key given: floor(a/b * k) by the
    score s, then the rest of the candidates by kappa (desc, position asc); ascending."""
    C = len(sg)
    k1 = (a * k) // b
    order1 = np.lexsort((np.arange(C), -sg))
    first = order1[:k1]
    mask = np.ones(C, dtype=bool)
    mask[first] = False
    rest = np.nonzero(mask)[0]
    order2 = np.lexsort((rest, -np.asarray(kg, dtype=np.float64)[rest]))
    return np.sort(np.concatenate([first, rest[order2[:k - k1]]]))


# ----------------------------------------------------------------------------
# Budget presets and re-eviction of a decoded cache.
# ----------------------------------------------------------------------------

def streaming_positions(C: int, k: int, sinks: int) -> np.ndarray:
    """StreamingLLM's kept candidates of one head with budget k (window not included): the
    first min(sinks, k) positions and the most recent k - min(sinks, k) before the window,
    ascending."""
    if k < 0 or k > C:
        raise ValueError("budget out of range")
    s = min(sinks, k)
    return np.concatenate([np.arange(s), np.arange(C - (k - s), C)]).astype(np.int64)


def reevict_rows(held: Sequence[int], s: np.ndarray, keep: int) -> np.ndarray:
    """Re-eviction of one head of a flat cache: `held` lists the positions of its rows in row
    order (-1 for a row appended by decoding, no prefill score; positions >= C are the
    window).  Rows without a candidate position always stay; the rest compete by the
    prefill score s (desc, position asc).  Returns the kept row indices, ascending; `keep`
    rows in all."""
    held = np.asarray(held, dtype=np.int64)
    C = len(s)
    cand = np.nonzero((held >= 0) & (held < C))[0]
    forced = np.nonzero(~((held >= 0) & (held < C)))[0]
    k = keep - len(forced)
    if k < 0 or k > len(cand):
        raise ValueError("budget out of range")
    order = np.lexsort((held[cand], -np.asarray(s, dtype=np.float64)[held[cand]]))
    return np.sort(np.concatenate([cand[order[:k]], forced]))
