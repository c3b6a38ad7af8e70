"""Named synthetic workloads and their seeded input generator.

This module holds shapes, budgets and random inputs only: none of the eviction
method's arithmetic lives here.  Both the CUDA path and the fp64 oracle read the
tensors it makes, so the two sides always see the same bytes.

The workloads stand in for the long-context evaluations of the Ada-KV notes
(Ruler 16K and LongBench, Llama-3.1-8B / Mistral-7B, "Experimental setup"), the
LAVa notes (Mistral-7B at up to 128K, "Latency and peak memory") and the
CriticalKV notes (40% budget, "Main experiments").  Neither the datasets nor the
model weights are used: the recipe below only reproduces their shapes and the
qualitative structure of real attention (sparse and dispersed heads, a sink at
position 0, a few heavy keys, heavy-tailed value norms).

Recipe, per (sequence, layer) unit, from a generator seeded by
``unit_seed(base_seed, seq, layer)``:

* Q_win [Hq, w, d] and K [Hkv, n, d] are N(0, 1).
* Each query head q gets a temperature tau_q, log-uniform in ``temp``; the
  window queries (and the decode queries) of head q are multiplied by tau_q.
* Sink: one unit vector u_g per KV head g.  Every window query of the group
  gets +2*u_g (before the temperature), and K[g, 0] += 3*sqrt(d)*u_g.
* ``heavy`` keys per KV head at seeded positions in [1, n-w) get
  K += 2*sqrt(d)*u_g.
* V is N(0, 1); with ``v_lognormal`` > 0 each row (g, j) is multiplied by
  exp(v_lognormal * zeta), zeta ~ N(0, 1).
* W_O (CriticalKV only) is N(0, 1/D), one [d, D] block per KV head.
* Decode step s: q ~ N(0,1)*tau_q, k_new, v_new ~ N(0, 1).

Values are drawn in fp32 and rounded once to the storage dtype.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    layers: int
    hq: int
    hkv: int
    d: int
    n: int
    w: int
    pool: int
    dtype: str                      # "bf16" or "f32"
    temp: tuple                     # (lo, hi) of the log-uniform head temperature
    heavy: int = 0                  # planted heavy keys per KV head
    v_lognormal: float = 0.0        # sigma of the per-row log-normal V scale
    mode: str = "ada"               # "ada", "lava" or "critical"
    group: str = "mean"             # GQA reduction: "mean" or "max"
    budget_kind: str = "layer"      # "layer": B per layer; "total": one total per sequence
    head_budget_frac: Optional[float] = None   # B = hkv*floor(frac*n)
    head_budget_tokens: Optional[int] = None   # B = hkv*tokens
    layer_budget: Optional[int] = None         # B given directly
    total_per_head_layer: Optional[int] = None # total = tokens*hkv*layers
    alpha: tuple = (1, 5)           # safeguard weight on the uniform share, as num/den
    crit_alpha: tuple = (1, 2)      # CriticalKV stage-1 fraction, as num/den
    crit_eps: float = 1e-6
    model_dim: int = 0              # D of W_O (CriticalKV only)
    decode_steps: int = 1
    reserve: int = 0                # flat-cache rows kept free per head for decode appends
    seed: int = 0xADA0

    @property
    def group_size(self) -> int:
        return self.hq // self.hkv

    @property
    def candidates(self) -> int:
        return self.n - self.w

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def layer_budget_value(self) -> int:
        """Layer budget B including the w*Hkv window rows (fixed-budget mode)."""
        if self.layer_budget is not None:
            return self.layer_budget
        if self.head_budget_tokens is not None:
            return self.hkv * self.head_budget_tokens
        if self.head_budget_frac is not None:
            return self.hkv * int(math.floor(self.head_budget_frac * self.n))
        raise ValueError("workload has no per-layer budget")

    def total_budget_value(self) -> int:
        """Total budget over all layers of one sequence (entropy mode)."""
        return self.total_per_head_layer * self.hkv * self.layers

    def budgets(self) -> torch.Tensor:
        """The int64 budget argument of kv_allocate: [batch, layers] or [batch]."""
        if self.budget_kind == "layer":
            return torch.full((self.batch, self.layers), self.layer_budget_value(),
                              dtype=torch.int64)
        return torch.full((self.batch,), self.total_budget_value(), dtype=torch.int64)

    def flat_capacity_rows(self) -> int:
        """Rows the flat K (or V) buffer needs for every (sequence, layer)."""
        if self.budget_kind == "layer":
            per_seq = self.layers * self.layer_budget_value()
        else:
            per_seq = self.total_budget_value()
        return self.batch * (per_seq + self.layers * self.hkv * self.reserve)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # Tiny single MHA layer, fp32: checked in full against the oracle.
    "tiny_mha_f32": Workload(
        name="tiny_mha_f32", batch=1, layers=1, hq=4, hkv=4, d=64, n=512, w=8, pool=7,
        dtype="f32", temp=(0.5, 8.0), heavy=3, layer_budget=128, reserve=1,
        decode_steps=1, seed=0xADA0 + 1),
    # Llama-3.1-8B-shaped single layer, 16K context, budget swept over 20/40/80% of n.
    "llama8b_16k_layer": Workload(
        name="llama8b_16k_layer", batch=1, layers=1, hq=32, hkv=8, d=128, n=16384, w=32,
        pool=7, dtype="bf16", temp=(0.5, 16.0), head_budget_frac=0.4, reserve=64,
        decode_steps=64, seed=0xADA0 + 2),
    # Full 32-layer Llama-3.1-8B-shaped KV set, batch 4, 32K context, 1024 per KV head.
    "llama8b_32k_b4": Workload(
        name="llama8b_32k_b4", batch=4, layers=32, hq=32, hkv=8, d=128, n=32768, w=32,
        pool=7, dtype="bf16", temp=(0.5, 16.0), head_budget_tokens=1024, reserve=256,
        decode_steps=256, seed=0xADA0 + 3),
    # Mistral-7B-shaped KV set, 128K context, LAVa scoring, total budget 128*Hkv*L.
    "mistral7b_128k_lava": Workload(
        name="mistral7b_128k_lava", batch=1, layers=32, hq=32, hkv=8, d=128, n=131072,
        w=32, pool=7, dtype="bf16", temp=(0.5, 16.0), v_lognormal=0.5, mode="lava",
        group="max", budget_kind="total", total_per_head_layer=128, alpha=(0, 1),
        reserve=128, decode_steps=128, seed=0xADA0 + 4),
    # CriticalKV on a Llama-3.1-8B-shaped stack, 64K context, 40% budget, D=4096.
    "llama8b_64k_criticalkv": Workload(
        name="llama8b_64k_criticalkv", batch=1, layers=32, hq=32, hkv=8, d=128, n=65536,
        w=32, pool=7, dtype="bf16", temp=(0.5, 16.0), mode="critical",
        head_budget_frac=0.4, model_dim=4096, reserve=64, decode_steps=64,
        seed=0xADA0 + 5),
}


def unit_seed(base_seed: int, seq: int, layer: int, stream: int = 0) -> int:
    """Deterministic per-(sequence, layer) seed (splitmix-style integer mix)."""
    x = (base_seed * 0x9E3779B97F4A7C15 + seq * 0xBF58476D1CE4E5B9
         + layer * 0x94D049BB133111EB + stream * 0xD6E8FEB86659FD93) & ((1 << 64) - 1)
    x ^= x >> 31
    x = (x * 0xBF58476D1CE4E5B9) & ((1 << 64) - 1)
    x ^= x >> 27
    return x & ((1 << 63) - 1)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_unit(wl: Workload, seq: int, layer: int, device="cpu") -> dict:
    """Prefill-side inputs of one (sequence, layer): q_win, k, v, tau (and w_o)."""
    dev = torch.device(device)
    g = _gen(dev, unit_seed(wl.seed, seq, layer))
    f32 = torch.float32
    hq, hkv, d, n, w, G = wl.hq, wl.hkv, wl.d, wl.n, wl.w, wl.group_size
    lo, hi = wl.temp
    u = torch.rand(hq, generator=g, device=dev, dtype=f32)
    tau = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    sink = torch.randn(hkv, d, generator=g, device=dev, dtype=f32)
    sink = sink / sink.norm(dim=1, keepdim=True)
    q = torch.randn(hq, w, d, generator=g, device=dev, dtype=f32)
    q += 2.0 * sink.repeat_interleave(G, dim=0)[:, None, :]
    q *= tau[:, None, None]
    k = torch.randn(hkv, n, d, generator=g, device=dev, dtype=f32)
    k[:, 0, :] += 3.0 * math.sqrt(d) * sink
    if wl.heavy > 0 and n - w > 1:
        for h in range(hkv):
            pos = torch.randint(1, n - w, (wl.heavy,), generator=g, device=dev)
            k[h, pos, :] += 2.0 * math.sqrt(d) * sink[h]
    v = torch.randn(hkv, n, d, generator=g, device=dev, dtype=f32)
    if wl.v_lognormal > 0:
        zeta = torch.randn(hkv, n, 1, generator=g, device=dev, dtype=f32)
        v *= torch.exp(wl.v_lognormal * zeta)
    out = {
        "q_win": q.to(wl.torch_dtype),
        "k": k.to(wl.torch_dtype),
        "v": v.to(wl.torch_dtype),
        "tau": tau,
    }
    if wl.mode == "critical":
        D = wl.model_dim
        wo = torch.randn(hkv, d, D, generator=g, device=dev, dtype=f32) / math.sqrt(D)
        out["w_o"] = wo.to(wl.torch_dtype)
    return out


def make_decode_step(wl: Workload, step: int, tau: torch.Tensor, seq: int, layer: int,
                     device="cpu") -> dict:
    """Decode-step inputs of one (sequence, layer): q [Hq, d], k_new, v_new [Hkv, d]."""
    dev = torch.device(device)
    g = _gen(dev, unit_seed(wl.seed, seq, layer, stream=1 + step))
    f32 = torch.float32
    q = torch.randn(wl.hq, wl.d, generator=g, device=dev, dtype=f32) * tau.to(dev)[:, None]
    kn = torch.randn(wl.hkv, wl.d, generator=g, device=dev, dtype=f32)
    vn = torch.randn(wl.hkv, wl.d, generator=g, device=dev, dtype=f32)
    return {"q": q.to(wl.torch_dtype), "k_new": kn.to(wl.torch_dtype),
            "v_new": vn.to(wl.torch_dtype)}


def make_batch(wl: Workload, device="cpu", seqs: Optional[Sequence[int]] = None,
               layers: Optional[Sequence[int]] = None) -> dict:
    """Stack units into the ABI layouts [B][L][...] for the chosen sequences/layers."""
    seqs = list(range(wl.batch)) if seqs is None else list(seqs)
    layers = list(range(wl.layers)) if layers is None else list(layers)
    B, L = len(seqs), len(layers)
    dt = wl.torch_dtype
    dev = torch.device(device)
    q_win = torch.empty(B, L, wl.hq, wl.w, wl.d, dtype=dt, device=dev)
    k = torch.empty(B, L, wl.hkv, wl.n, wl.d, dtype=dt, device=dev)
    v = torch.empty(B, L, wl.hkv, wl.n, wl.d, dtype=dt, device=dev)
    tau = torch.empty(B, L, wl.hq, dtype=torch.float32, device=dev)
    w_o = None
    if wl.mode == "critical":
        w_o = torch.empty(L, wl.hkv, wl.d, wl.model_dim, dtype=dt, device=dev)
    for bi, s in enumerate(seqs):
        for li, l in enumerate(layers):
            u = make_unit(wl, s, l, device=dev)
            q_win[bi, li] = u["q_win"]
            k[bi, li] = u["k"]
            v[bi, li] = u["v"]
            tau[bi, li] = u["tau"]
            if w_o is not None and bi == 0:
                w_o[li] = u["w_o"]
            del u
    return {"q_win": q_win, "k": k, "v": v, "tau": tau, "w_o": w_o}


def make_decode_batch(wl: Workload, step: int, tau: torch.Tensor, device="cpu",
                      seqs: Optional[Sequence[int]] = None,
                      layers: Optional[Sequence[int]] = None) -> dict:
    """Decode inputs for every (sequence, layer): q [B][L][Hq][d], k_new/v_new [B][L][Hkv][d]."""
    seqs = list(range(wl.batch)) if seqs is None else list(seqs)
    layers = list(range(wl.layers)) if layers is None else list(layers)
    B, L = len(seqs), len(layers)
    dev = torch.device(device)
    dt = wl.torch_dtype
    q = torch.empty(B, L, wl.hq, wl.d, dtype=dt, device=dev)
    kn = torch.empty(B, L, wl.hkv, wl.d, dtype=dt, device=dev)
    vn = torch.empty(B, L, wl.hkv, wl.d, dtype=dt, device=dev)
    for bi, s in enumerate(seqs):
        for li, l in enumerate(layers):
            st = make_decode_step(wl, step, tau[bi, li], s, l, device=dev)
            q[bi, li] = st["q"]
            kn[bi, li] = st["k_new"]
            vn[bi, li] = st["v_new"]
    return {"q": q, "k_new": kn, "v_new": vn}


def make_flat_cache(wl: Workload, mean_len: int, sigma: float, reserve: int, seed: int,
                    device="cpu") -> dict:
    """A flat cache laid out as kv_compact writes it, for decode-only measurements.

    Per-head lengths are log-normal (sigma) around mean_len, at least wl.w (the window
    rows every head keeps), each head followed by `reserve` free rows; K, V, q, k_new and
    v_new are N(0, 1) in the storage dtype.  Returns cu [B][L][Hkv+1], lens [B][L][Hkv],
    k_flat / v_flat [cap][d], q [B][L][Hq][d], k_new / v_new [B][L][Hkv][d] and cap.
    """
    dev = torch.device(device)
    g = _gen(torch.device("cpu"), seed)
    B, L, hkv = wl.batch, wl.layers, wl.hkv
    H = B * L * hkv
    f = torch.exp(torch.randn(H, generator=g) * sigma)
    lens = (f / f.mean() * mean_len).round().clamp(min=wl.w).to(torch.int64)
    ext = lens + reserve
    flat = torch.cat([torch.zeros(1, dtype=torch.int64), ext.cumsum(0)])
    cu = torch.stack([flat[s * hkv: s * hkv + hkv + 1] for s in range(B * L)])
    cap = int(flat[-1])
    dt = wl.torch_dtype
    gd = _gen(dev, seed + 1)
    out = {
        "cu": cu.reshape(B, L, hkv + 1).to(dev),
        "lens": lens.to(torch.int32).reshape(B, L, hkv).to(dev),
        "k_flat": torch.randn(cap, wl.d, generator=gd, device=dev).to(dt),
        "v_flat": torch.randn(cap, wl.d, generator=gd, device=dev).to(dt),
        "q": torch.randn(B, L, wl.hq, wl.d, generator=gd, device=dev).to(dt),
        "k_new": torch.randn(B, L, hkv, wl.d, generator=gd, device=dev).to(dt),
        "v_new": torch.randn(B, L, hkv, wl.d, generator=gd, device=dev).to(dt),
        "cap": cap,
    }
    return out
