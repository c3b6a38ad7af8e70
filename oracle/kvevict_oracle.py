"""Plain fp64 CPU oracle of head-adaptive KV-cache eviction and flat decode attention.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The library path never does: it shares no code, header, table or helper
with the CUDA kernels.  Every function is written from the definitions on the
method's pages, as loops or single library primitives (a matmul, a sort), with no
blocking or fusion.

Pages (cited by title and section):

* "Ada-KV: Optimizing KV Cache Eviction by Adaptive Budget Allocation for
  Efficient LLM Inference" -- papercache notes (Chinese) and the arXiv HTML.
  Formal model of multi-head self-attention, Eviction Decision and post-eviction
  output, Theorems 3.1-3.3, Algorithm 1 (adaptive budget allocation),
  Algorithm 2 (integration into SnapKV), the flat-cache / GQA remarks.
* "LAVa: Layer-wise KV Cache Eviction with Dynamic Budget Allocation" --
  Definition 1 (LAVa score), Theorem 1, head-flattened layer-wise eviction,
  uncertainty-based layer budgets, GQA adaptation.
* "CriticalKV: Optimizing KV Cache Eviction from an Output Perturbation
  Perspective" -- key designs: the perturbation bound and the two-stage greedy
  selection, used as a plug-in of Ada-KV.
* The LaProx page ("Reformulating KV cache eviction for long-context LLM
  inference"), Eq. 2, for the 1/sqrt(d_h) logit scale.

Readings taken where the pages are silent or disagree:

* Logits carry 1/sqrt(d_h) (LaProx Eq. 2, LAVa's residual-stream view); the
  Ada-KV arXiv page leaves the scale out only to keep its notation short.
* The window softmax normalises over all n keys with the causal mask: window
  row t is the query of position n-w+t and sees keys j <= n-w+t.  The literal
  prefix-only normalisation of Algorithm 2 is kept as ``normalise="prefix"``.
* Scores are the window MEAN (= sum / w), then a stride-1 max-pool of width
  ``pool`` clipped to the candidate range [0, n-w), then the GQA group
  reduction (mean for Ada-KV, max for LAVa).  Pooling each window row before the
  mean (the literal Algorithm 2 order) is kept as ``order="pool_rows"``.
* GQA maps query head q to KV head floor(q / G).
* The layer budget B counts the w*Hkv window rows (Ada-KV Algorithm 2 takes the
  window's rows off the budget before allocating); B' = B - w*Hkv is what the
  selection distributes.
* Safeguard: B_g = alpha*B'/Hkv + (1-alpha)*f_g, alpha the weight on the
  uniform share (alpha = 1 gives uniform SnapKV, budgets never fall below
  floor(alpha*B'/Hkv)); alpha = a/b is rational and rounding is exact.
* Ties in every Top-k follow total orders: (score desc, head asc, position asc)
  layer-wide, (score desc, position asc) per head.
"""
from __future__ import annotations

import math
from typing import List, Optional, Sequence, Tuple

import numpy as np

__all__ = [
    "window_logits", "row_softmax", "window_attention", "window_reduce", "max_pool",
    "group_reduce", "v_l1_max", "critical_row_norm", "score_layer",
    "global_topk_counts", "safeguard_blend", "head_budgets",
    "layer_entropy", "lava_layer_budgets", "topk_positions", "critical_positions",
    "compact_layer", "flat_decode", "dense_decode", "masked_head_output",
    "eviction_bound", "retained_mass", "lava_bound",
]


# ----------------------------------------------------------------------------
# Scoring.  Ada-KV Algorithm 2 (observation-window scoring), LAVa Definition 1,
# CriticalKV's projected-value norm.
# ----------------------------------------------------------------------------

def window_logits(q_win: np.ndarray, k: np.ndarray, scale: float,
                  causal: bool = True) -> np.ndarray:
    """z[q, t, j] = q_win[q, t] . k[g(q), j] * scale, masked to -inf above the diagonal.

    q_win [Hq, w, d], k [Hkv, n, d] -> z [Hq, w, n].  Ada-KV Algorithm 2 forms
    Q_win K^T per head; the logit scale is the 1/sqrt(d_h) of LaProx Eq. 2.  The
    window query t belongs to position n-w+t and so sees keys j <= n-w+t.
    """
    hq, w, d = q_win.shape
    hkv, n, _ = k.shape
    G = hq // hkv
    z = np.empty((hq, w, n), dtype=np.float64)
    for q in range(hq):
        g = q // G
        z[q] = (q_win[q].astype(np.float64) @ k[g].astype(np.float64).T) * scale
    if causal:
        for t in range(w):
            z[:, t, n - w + t + 1:] = -np.inf
    return z


def row_softmax(z: np.ndarray) -> np.ndarray:
    """softmax over the last axis: exp(z - max) / sum(exp(z - max))."""
    m = np.max(z, axis=-1, keepdims=True)
    e = np.exp(z - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def window_attention(q_win, k, scale, normalise: str = "causal_all") -> np.ndarray:
    """Window attention probabilities P [Hq, w, n] (Ada-KV Algorithm 2, first step).

    ``causal_all``: each row is a real attention row, normalised over every key it
    can see.  ``prefix``: the literal reading, softmax over the keys outside the
    window only (columns >= n-w come back as zero).
    """
    n = k.shape[1]
    w = q_win.shape[1]
    z = window_logits(q_win, k, scale, causal=True)
    if normalise == "causal_all":
        return row_softmax(z)
    if normalise == "prefix":
        zp = z.copy()
        zp[:, :, n - w:] = -np.inf
        return row_softmax(zp)
    raise ValueError(normalise)


def max_pool(a: np.ndarray, pool: int) -> np.ndarray:
    """Stride-1, same-length 1-D max-pool along the last axis, window clipped to the ends.

    p[..., j] = max over k in [j - pool//2, j + pool//2] intersected with [0, C) of a[..., k].
    """
    C = a.shape[-1]
    r = pool // 2
    p = np.empty_like(a)
    for j in range(C):
        lo, hi = max(0, j - r), min(C, j + r + 1)
        p[..., j] = np.max(a[..., lo:hi], axis=-1)
    return p


def window_reduce(P: np.ndarray, C: int, pool: int, order: str = "mean_then_pool") -> np.ndarray:
    """Per query head score over the candidates j < C (Ada-KV Algorithm 2, pooling step).

    ``mean_then_pool``: a[q, j] = (1/w) sum_t P[q, t, j], then max_pool.
    ``pool_rows``: max_pool each window row first, then the mean over t.
    """
    if C == 0:
        return np.zeros((P.shape[0], 0))
    Pc = P[:, :, :C]
    if order == "mean_then_pool":
        return max_pool(Pc.mean(axis=1), pool)
    if order == "pool_rows":
        return max_pool(Pc, pool).mean(axis=1)
    raise ValueError(order)


def group_reduce(p: np.ndarray, hkv: int, how: str) -> np.ndarray:
    """GQA: the KV-head score is the mean (Ada-KV GQA remark) or the max (LAVa GQA
    adaptation) of its query heads' scores.  p [Hq, C] -> s [Hkv, C]."""
    hq = p.shape[0]
    G = hq // hkv
    s = np.empty((hkv, p.shape[1]))
    for g in range(hkv):
        block = p[g * G:(g + 1) * G]
        if how == "mean":
            s[g] = block.mean(axis=0)
        elif how == "max":
            s[g] = block.max(axis=0)
        else:
            raise ValueError(how)
    return s


def v_l1_max(v: np.ndarray) -> np.ndarray:
    """LAVa's head constant  Vbar[g] = max over k of ||V[g, k]||_1  (Theorem 1 / Definition 1)."""
    return np.abs(v.astype(np.float64)).sum(axis=2).max(axis=1)


def critical_row_norm(v: np.ndarray, w_o: np.ndarray, C: int) -> np.ndarray:
    """CriticalKV's projected-value norm  c[g, j] = ||(V W^O)_j||_1  for j < C.

    v [Hkv, n, d], w_o [Hkv, d, D] (one output block per KV head) -> [Hkv, C].
    """
    hkv = v.shape[0]
    c = np.empty((hkv, C))
    for g in range(hkv):
        proj = v[g, :C].astype(np.float64) @ w_o[g].astype(np.float64)
        c[g] = np.abs(proj).sum(axis=1)
    return c


def score_layer(q_win, k, v, *, w: int, pool: int, mode: str = "ada", group: str = "mean",
                w_o=None, scale: Optional[float] = None, normalise: str = "causal_all",
                order: str = "mean_then_pool") -> Tuple[np.ndarray, Optional[np.ndarray]]:
    """Scores of one (sequence, layer).  Returns (s [Hkv, C], c [Hkv, C] or None).

    ada:      s = group_reduce(max_pool(window mean of P))                (Ada-KV Alg. 2)
    lava:     s = Vbar[g] * group_max(max_pool(window mean of P))         (LAVa Def. 1, GQA)
    critical: s as ada, plus c = ||(V W^O)_j||_1                          (CriticalKV)
    """
    hq, _, d = q_win.shape
    hkv, n, _ = k.shape
    C = n - w
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    P = window_attention(q_win, k, scale, normalise=normalise)
    p = window_reduce(P, C, pool, order=order)
    s = group_reduce(p, hkv, group)
    c = None
    if mode == "lava":
        s = s * v_l1_max(v)[:, None]
    elif mode == "critical":
        c = critical_row_norm(v, w_o, C)
    elif mode != "ada":
        raise ValueError(mode)
    return s, c


# ----------------------------------------------------------------------------
# Allocation.  Ada-KV Algorithm 1 and the safeguard of Algorithm 2; LAVa's
# head-flattened layer eviction and uncertainty-based layer budgets.
# ----------------------------------------------------------------------------

def global_topk_counts(s: np.ndarray, Bp: int) -> np.ndarray:
    """Ada-KV Algorithm 1: concatenate all heads' scores, take the top B', count per head.

    Order: score descending, then head ascending, then position ascending.
    """
    hkv, C = s.shape
    flat = s.reshape(-1)
    heads = np.repeat(np.arange(hkv), C)
    pos = np.tile(np.arange(C), hkv)
    order = np.lexsort((pos, heads, -flat))
    chosen = order[:Bp]
    return np.bincount(heads[chosen], minlength=hkv).astype(np.int64)


def safeguard_blend(f: Sequence[int], Bp: int, a: int, b: int) -> np.ndarray:
    """Blend the adaptive counts with the uniform share, alpha = a/b on the uniform side.

    B_g = floor(X_g / (b*H)) with X_g = a*B' + (b-a)*H*f_g, then the B' - sum B_g
    leftover units go one each to the heads with the largest X_g mod (b*H),
    ties to the lower head.  Exact integers throughout.
    """
    H = len(f)
    den = b * H
    X = [a * Bp + (b - a) * H * int(fg) for fg in f]
    Bg = [x // den for x in X]
    rem = [x % den for x in X]
    left = Bp - sum(Bg)
    for g in sorted(range(H), key=lambda h: (-rem[h], h))[:left]:
        Bg[g] += 1
    return np.array(Bg, dtype=np.int64)


def head_budgets(s: np.ndarray, B: int, w: int, a: int, b: int) -> Tuple[np.ndarray, np.ndarray]:
    """Per-head budgets of one layer: (f, B_g), with sum B_g = B' = B - w*Hkv.

    Ada-KV Algorithm 2: remove the window rows from the layer budget, run
    Algorithm 1 on the scores, apply the safeguard.
    """
    hkv, C = s.shape
    Bp = B - w * hkv
    if Bp < 0 or Bp > hkv * C:
        raise ValueError("budget out of range")
    f = global_topk_counts(s, Bp)
    return f, safeguard_blend(f, Bp, a, b)


def layer_entropy(s: np.ndarray, n: int) -> float:
    """LAVa's layer uncertainty e_l = -sum_{h,i} shat log shat / (H * N), shat = s / sum s.

    The sum runs over the candidate scores of every KV head of the layer; 0 log 0 = 0.
    """
    hkv = s.shape[0]
    flat = s.reshape(-1).astype(np.float64)
    tot = flat.sum()
    if tot <= 0.0:
        return 0.0
    sh = flat / tot
    nz = sh[sh > 0]
    return float(-(nz * np.log(nz)).sum() / (hkv * n))


def lava_layer_budgets(e: Sequence[float], total: int, w: int, hkv: int, C: int) -> np.ndarray:
    """LAVa layer budgets: the selectable total split in proportion to e_l.

    R = total - L*w*Hkv.  Layers whose share exceeds Hkv*C are capped and the rest
    re-split; the others get floor(R_rem * e_l / sum e) plus one each for the
    largest fractional parts (ties to the lower layer).  If every e_l is zero the
    split is uniform.  Returns B_l including the w*Hkv window rows.
    """
    L = len(e)
    R = total - L * w * hkv
    cap = hkv * C
    if R < 0 or R > L * cap:
        raise ValueError("total budget out of range")
    from fractions import Fraction
    ef = [Fraction(float(x)) for x in e]
    sel = [None] * L
    active = list(range(L))
    rem = R
    while True:
        esum = sum(ef[l] for l in active)
        quota = {}
        for l in active:
            quota[l] = (Fraction(rem) * ef[l] / esum) if esum > 0 else Fraction(rem, len(active))
        over = [l for l in active if quota[l] > cap]
        if not over:
            break
        for l in over:
            sel[l] = cap
            rem -= cap
        active = [l for l in active if l not in over]
    fl = {l: math.floor(quota[l]) for l in active}
    for l in active:
        sel[l] = fl[l]
    left = rem - sum(fl.values())
    for l in sorted(active, key=lambda x: (-(quota[x] - fl[x]), x))[:left]:
        sel[l] += 1
    return np.array([x + w * hkv for x in sel], dtype=np.int64)


# ----------------------------------------------------------------------------
# Selection and the flat cache.  Ada-KV Algorithm 2 (per-head Top-k, keep the
# window), the flat layout remark; CriticalKV two-stage greedy selection.
# ----------------------------------------------------------------------------

def topk_positions(sg: np.ndarray, k: int) -> np.ndarray:
    """Positions of the k largest scores of one head, (score desc, position asc), ascending."""
    C = len(sg)
    order = np.lexsort((np.arange(C), -sg))
    return np.sort(order[:k])


def critical_positions(sg: np.ndarray, cg: np.ndarray, k: int, a: int, b: int, eps: float,
                       kappa_dtype=np.float64) -> np.ndarray:
    """CriticalKV two-stage selection of k positions of one head, ascending.

    Stage 1 keeps the floor(a/b * k) largest by the attention score s.  Stage 2
    keeps the remaining k - k1 of the rest by kappa = (s + eps) * c.
    ``kappa_dtype`` is the precision kappa is formed in.
    """
    C = len(sg)
    k1 = (a * k) // b
    first = topk_positions(sg, k1)
    mask = np.ones(C, dtype=bool)
    mask[first] = False
    rest = np.nonzero(mask)[0]
    sk = np.asarray(sg, dtype=kappa_dtype)
    ck = np.asarray(cg, dtype=kappa_dtype)
    kappa = (sk + kappa_dtype(eps)) * ck
    kr = kappa[rest].astype(np.float64)
    order = np.lexsort((rest, -kr))
    second = rest[order[:k - k1]]
    return np.sort(np.concatenate([first, second]))


def compact_layer(k: np.ndarray, v: np.ndarray, s: np.ndarray, Bg: Sequence[int], w: int,
                  reserve: int = 0, c: Optional[np.ndarray] = None,
                  crit: Optional[Tuple[int, int, float]] = None, kappa_dtype=np.float64):
    """Retained cache of one layer in the flat layout (Ada-KV Algorithm 2, flat-cache remark).

    For each head g: kept_g = ascending selected positions followed by the window
    [C, n).  The heads are laid out back to back; head g owns rows
    [cu[g], cu[g+1]) with cu[g+1] = cu[g] + B_g + w + reserve, of which the first
    lens[g] = B_g + w are filled.  Returns (kept list, cu, lens, K_f, V_f).
    """
    hkv, n, d = k.shape
    C = n - w
    kept: List[np.ndarray] = []
    for g in range(hkv):
        if crit is None:
            sel = topk_positions(s[g], int(Bg[g]))
        else:
            a, b, eps = crit
            sel = critical_positions(s[g], c[g], int(Bg[g]), a, b, eps, kappa_dtype)
        kept.append(np.concatenate([sel, np.arange(C, n)]).astype(np.int64))
    lens = np.array([len(x) for x in kept], dtype=np.int64)
    cu = np.zeros(hkv + 1, dtype=np.int64)
    for g in range(hkv):
        cu[g + 1] = cu[g] + lens[g] + reserve
    Kf = np.zeros((cu[-1], d), dtype=np.float64)
    Vf = np.zeros((cu[-1], d), dtype=np.float64)
    for g in range(hkv):
        for r, j in enumerate(kept[g]):
            Kf[cu[g] + r] = k[g, j]
            Vf[cu[g] + r] = v[g, j]
    return kept, cu, lens, Kf, Vf


# ----------------------------------------------------------------------------
# Decode.  Ada-KV formal model: append k, v to the cache, then
# A_i = softmax(q_i K_i^T * scale) and the head output A_i V_i.
# ----------------------------------------------------------------------------

def flat_decode(q: np.ndarray, Kf: np.ndarray, Vf: np.ndarray, cu, lens, scale: float,
                k_new: Optional[np.ndarray] = None, v_new: Optional[np.ndarray] = None):
    """One decode step over the flat cache of one layer.  q [Hq, d] -> o [Hq, d].

    If k_new/v_new [Hkv, d] are given they are written at row cu[g] + lens[g]
    first and lens grows by one (the new token attends to itself).  Returns
    (o, Kf, Vf, lens) with the updated copies.
    """
    hq, d = q.shape
    hkv = len(lens)
    G = hq // hkv
    Kf = Kf.copy()
    Vf = Vf.copy()
    lens = np.array(lens, dtype=np.int64).copy()
    if k_new is not None:
        for g in range(hkv):
            r = cu[g] + lens[g]
            if r >= cu[g + 1]:
                raise ValueError("no reserve row left for the append")
            Kf[r] = k_new[g]
            Vf[r] = v_new[g]
            lens[g] += 1
    o = np.zeros((hq, d))
    for qh in range(hq):
        g = qh // G
        rows = slice(cu[g], cu[g] + lens[g])
        if lens[g] == 0:
            continue
        zz = Kf[rows] @ q[qh].astype(np.float64) * scale
        a = row_softmax(zz)
        o[qh] = a @ Vf[rows]
    return o, Kf, Vf, lens


def dense_decode(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Full-cache attention of one decode query per head.  q [Hq, d], K/V [Hkv, N, d]."""
    hq, d = q.shape
    hkv = K.shape[0]
    G = hq // hkv
    o = np.zeros((hq, d))
    for qh in range(hq):
        g = qh // G
        a = row_softmax(K[g].astype(np.float64) @ q[qh].astype(np.float64) * scale)
        o[qh] = a @ V[g].astype(np.float64)
    return o


# ----------------------------------------------------------------------------
# The pages' bounds, used to pin the oracle (Ada-KV Theorems 3.1-3.3, LAVa Theorem 1).
# ----------------------------------------------------------------------------

def masked_head_output(A: np.ndarray, T: np.ndarray, VW: np.ndarray) -> np.ndarray:
    """Ada-KV post-eviction output  yhat = sum_i (T_i * A_i / ||A_i * T_i||_1) V_i W_i^O.

    A, T [h, n]; VW [h, n, D] (the per-head product V_i W_i^O).
    """
    y = np.zeros(VW.shape[2])
    for i in range(A.shape[0]):
        m = A[i] * T[i]
        y += (m / m.sum()) @ VW[i]
    return y


def eviction_bound(A: np.ndarray, T: np.ndarray, Cmax: float) -> float:
    """Ada-KV Theorem 3.1:  eps = 2hC - 2C sum_i sum_j T_i^j A_i^j."""
    h = A.shape[0]
    return 2.0 * h * Cmax - 2.0 * Cmax * float((T * A).sum())


def retained_mass(s: np.ndarray, Bg: Sequence[int]) -> float:
    """Sum over heads of the B_g largest scores of each head (the sum T*A of Theorem 3.2)."""
    tot = 0.0
    for g in range(s.shape[0]):
        tot += float(np.sort(s[g])[::-1][:int(Bg[g])].sum())
    return tot


def lava_bound(A: np.ndarray, T: np.ndarray, vbar: np.ndarray, w_o: np.ndarray) -> float:
    """LAVa Theorem 1:  2 * ||W_O^T||_1 * sum_h sum_i A_h[i] * Vbar_h * (1 - T_h[i]).

    ||W_O^T||_1 is the largest absolute row sum of W_O (the induced 1-norm of W_O^T).
    """
    chat = float(np.abs(w_o).sum(axis=1).max())
    return 2.0 * chat * float((A * vbar[:, None] * (1.0 - T)).sum())
