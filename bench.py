#!/usr/bin/env python3
"""Throughput of the KV-cache eviction pass and the flat decode attention on GB300.

One step = one pass of the whole hot path over one batch: an eviction pass over every
(sequence, layer) of the workload (kv_score -> kv_allocate -> kv_compact) followed by one
decode step of flat_decode_attn over every layer (with the append).  The headline value is
eviction-pass prefix tokens per second per layer, (batch * n * L) / step_time / L, i.e.
batch * n / step_time summed over ranks: the prompt tokens whose whole-model cache the path
evicts (and then decodes over) per second.  `eviction_only` gives the same rate over the
eviction stages alone (score + allocate + compact).  The second number, the flat varlen
decode attention's HBM GB/s, is measured on its own with L2 flushed before every decode
step.  The other workloads of the pages' configurations are timed after the headline one
(`workloads`), and the CPU oracle on the host cores (`cpu_baseline`: one core and all).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the only other implementation of the
method there is) on a bounded sample of the same workload.
"""
from __future__ import annotations

import os

# The CPU oracle is timed single-threaded; pin the BLAS pools before numpy loads.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import json
import math
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "eviction-pass prefix tokens/s per layer; flat varlen decode attn HBM GB/s"
UNIT = "tokens/s/layer"
DEFAULT_WORKLOAD = "mistral7b_128k_lava"
L2_BYTES = 129 * 1024 * 1024


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--layers", type=int, default=0,
                    help="override the workload's layer count (profiling cases)")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--decode-steps", type=int, default=-1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-batches", default="",
                    help="comma-separated batch sizes: decode alone over that many replicas of "
                         "the evicted sequence's flat cache (e.g. 1,8,32)")
    ap.add_argument("--decode-only", action="store_true",
                    help="decode alone on a synthetic flat cache shaped like the workload's "
                         "(log-normal head lengths around its mean budget per head); no "
                         "eviction inputs are built")
    ap.add_argument("--decode-sigma", type=float, default=0.4,
                    help="--decode-only: sigma of the log-normal head lengths (0.4 matches the "
                         "spread of the 128K LAVa allocation: p90 1.5x, max 2.8x the mean)")
    ap.add_argument("--no-decode-per-layer", action="store_true",
                    help="skip the decode-only measurement with one call per layer")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the step with eager launches only (no CUDA graph replay)")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the step timings of the pages' other configurations")
    ap.add_argument("--no-decode-large", action="store_true",
                    help="skip the decode-only measurement on the large flat cache")
    return ap.parse_args()


def rank_sequences(rank: int, batch: int) -> range:
    """The sequences rank `rank` evicts: each rank owns `batch` sequences of its own (weak
    scaling, no data-path exchange)."""
    return range(rank * batch, (rank + 1) * batch)


def max_over_ranks(t: float, device=None) -> float:
    """The slowest rank's time (all ranks get it); the local time when not distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return t
    tt = torch.tensor([t], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def aggregate_value(world: int, batch: int, n: int, layers: int, ms: float) -> float:
    """Whole-job eviction-pass prefix tokens/s per layer: every rank's batch * n * L
    (token, layer) pairs in the slowest rank's step time, per layer (divided by L)."""
    return world * batch * n * layers / (ms / 1e3) / layers


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "score_tc_kernel_traffic.txt")
TRAFFIC_SOURCES = ("kv_cache_eviction_gb300/csrc/score_tc.cu",
                   "kv_cache_eviction_gb300/csrc/tc_ptx.cuh")


def score_kernel_sha():
    import hashlib
    h = hashlib.sha256()
    for rel in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def read_traffic(workload: str):
    """DRAM bytes of one score_tc_kernel launch of `workload` from the committed ncu
    summary, or None when there is none or the kernel's source changed since."""
    try:
        kv = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256") != score_kernel_sha():
            return None
        if kv.get("workload") != workload:
            return None
        return int(kv["bytes_per_launch"])
    except Exception:
        return None


def read_tensor_peak():
    """Sustained dense bf16 TFLOP/s (the norm kernel runs inside a long step)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops_sustained"]), "measured (sustained)"
    except Exception:
        return 1700.0, "fallback (sustained)"


def read_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# CPU oracle sample (the cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def oracle_heads(wl, count: int, use_cuda_inputs: bool):
    """Inputs of `count` KV heads as fp64 numpy arrays: (sequence 0, layer l, head g) in
    (l, g) order, each with its G window queries, its K and V rows (and its W_O block) and
    one decode step's q, k_new and v_new."""
    import torch
    from kv_cache_eviction_gb300 import workloads as W
    dev = "cuda" if use_cuda_inputs else "cpu"
    G = wl.hq // wl.hkv
    to = lambda t: t.to("cpu", torch.float64).numpy()
    out = []
    layer = 0
    while len(out) < count:
        u = W.make_unit(wl, 0, layer, device=dev)
        dec = W.make_decode_step(wl, 0, u["tau"], 0, layer, device=dev)
        for g in range(wl.hkv):
            if len(out) == count:
                break
            x = {"q": to(u["q_win"][g * G:(g + 1) * G]), "k": to(u["k"][g:g + 1]),
                 "v": to(u["v"][g:g + 1]), "dq": to(dec["q"][g * G:(g + 1) * G]),
                 "kn": to(dec["k_new"][g:g + 1]), "vn": to(dec["v_new"][g:g + 1])}
            if "w_o" in u:
                x["w_o"] = to(u["w_o"][g:g + 1])
            out.append(x)
        del u, dec
        layer += 1
    return out


def oracle_step(wl, x):
    """The oracle's eviction of one KV head (score, its uniform share of the layer budget,
    selection, gather) plus one decode step of its G query heads."""
    import numpy as np
    import oracle as O
    s, c = O.score_layer(x["q"], x["k"], x["v"], w=wl.w, pool=wl.pool, mode=wl.mode,
                         group=wl.group, w_o=x.get("w_o"))
    if wl.budget_kind == "layer":
        Bl = wl.layer_budget_value()
    else:
        Bl = wl.total_budget_value() // wl.layers
    Bp = (Bl - wl.w * wl.hkv) // wl.hkv
    f, Bg = O.head_budgets(s, Bp + wl.w, wl.w, wl.alpha[0], wl.alpha[1])
    crit = (wl.crit_alpha[0], wl.crit_alpha[1], wl.crit_eps) if wl.mode == "critical" else None
    kept, cu, lens, Kf, Vf = O.compact_layer(x["k"], x["v"], s, Bg, wl.w, reserve=1, c=c,
                                             crit=crit)
    o, *_ = O.flat_decode(x["dq"], Kf, Vf, cu, lens, 1.0 / math.sqrt(wl.d), x["kn"], x["vn"])
    return float(np.abs(o).sum())


def oracle_rate(wl, heads: int, seconds: float) -> float:
    """tokens/s per layer of the oracle: `heads` KV heads of n prefix tokens are each
    1 / (L * Hkv) of a sequence's whole-model eviction."""
    return heads * wl.n / (wl.layers * wl.hkv * seconds)


def sample_desc(wl, heads=1):
    return ("%d KV head(s) of (sequence 0, layers 0..%d) of %s (n=%d, %d query heads each): "
            "window scoring, the head's uniform share of the layer budget, selection, gather "
            "and one decode step; tokens/s per layer = heads * n / (L * Hkv * time)" %
            (heads, (heads - 1) // wl.hkv, wl.name, wl.n, wl.hq // wl.hkv))


_POOL_WL = None
_POOL_X = None


def _oracle_worker(i):
    t0 = time.perf_counter()
    oracle_step(_POOL_WL, _POOL_X[i])
    return time.perf_counter() - t0


def cpu_baseline(wl):
    """The oracle on the host: one KV head on one core, then one head per core on every core
    at once (a process pool forked before the process touches the GPU).  Call it before any
    CUDA work."""
    import multiprocessing
    global _POOL_WL, _POOL_X
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    nproc = os.cpu_count() or cores
    _POOL_WL = wl
    _POOL_X = oracle_heads(wl, cores, False)
    # one core: heads one after another, until about 10 s of work or every generated head
    t1, done = 0.0, 0
    while done < cores and (done == 0 or t1 < 10.0):
        t1 += _oracle_worker(done)
        done += 1
    res = {"value": oracle_rate(wl, done, t1), "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": sample_desc(wl, done), "seconds": t1, "nproc": nproc}
    if cores > 1:
        with multiprocessing.get_context("fork").Pool(cores) as pool:
            pool.map(_oracle_worker, range(cores), chunksize=1)    # touch every worker once
            t0 = time.perf_counter()
            per = pool.map(_oracle_worker, range(cores), chunksize=1)
            t_all = time.perf_counter() - t0
        res["all_cores"] = {"value": oracle_rate(wl, cores, t_all), "unit": UNIT,
                            "cores": cores, "seconds": t_all,
                            "sample": sample_desc(wl, cores),
                            "per_head_seconds_mean": statistics.mean(per)}
    _POOL_X = None
    return res


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return 0
    import torch
    from kv_cache_eviction_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]
    if args.layers > 0:
        wl = wl.with_(layers=args.layers)
    use_cuda = torch.cuda.is_available()
    if use_cuda:
        torch.cuda.set_device(local)
    x = oracle_heads(wl, 1, use_cuda)[0]
    for _ in range(args.warmup):
        oracle_step(wl, x)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(wl, x)
        times.append(time.perf_counter() - t0)
    t = statistics.mean(times)
    value = oracle_rate(wl, 1, t)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generator)",
        "config": {"workload": wl.name, "sample": "1 KV head of 1 (sequence, layer)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample_desc(wl, 1), "nproc": os.cpu_count()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.3)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def algorithmic_bytes(wl, B, L, head_budget_total_rows, decode_rows):
    """Bytes each stage must move: K once (and V once for LAVa and CriticalKV, plus W_O for
    CriticalKV), the window queries and the scores written (score); the scores read
    (allocate); the scores read, the kept K/V rows read and written and their indices
    (compact); every used K/V row, q, out, k_new and v_new (decode)."""
    e = wl.elem_bytes
    C = wl.n - wl.w
    kv_bytes = B * L * wl.hkv * wl.n * wl.d * e
    q_bytes = B * L * wl.hq * wl.w * wl.d * e
    s_bytes = B * L * wl.hkv * C * 4
    score = kv_bytes + q_bytes + s_bytes
    if wl.mode in ("lava", "critical"):
        score += kv_bytes
    if wl.mode == "critical":
        score += L * wl.hkv * wl.d * wl.model_dim * e + s_bytes
    allocate = s_bytes
    row = wl.d * e
    compact = s_bytes + 4 * head_budget_total_rows * row + 4 * head_budget_total_rows
    if wl.mode == "critical":
        compact += s_bytes
    decode = 2 * decode_rows * row + 2 * B * L * wl.hq * wl.d * e + 4 * B * L * wl.hkv * wl.d * e
    return {"score": score, "allocate": allocate, "compact": compact, "decode": decode}


def decode_batches(kv, W, wl, dev, stream, flush, kf, vf, cu, lens, cap, batches, steps=3):
    """flat_decode_attn alone over b copies of one evicted sequence's flat cache, for each b in
    `batches`.  The copies sit at distinct addresses of one flat buffer (offsets shifted by
    the sequence's capacity), with fresh q / k_new / v_new per sequence; L2 flushed before
    each step.  Replicas stand in for b independently evicted sequences."""
    import torch
    res = []
    L, hkv = wl.layers, wl.hkv
    for b in batches:
        shape_b = kv.KvShape.from_workload(wl.with_(batch=b))
        kf_b = torch.empty(b * cap, wl.d, dtype=kf.dtype, device=dev)
        vf_b = torch.empty_like(kf_b)
        for i in range(b):
            kf_b[i * cap:(i + 1) * cap].copy_(kf[:cap])
            vf_b[i * cap:(i + 1) * cap].copy_(vf[:cap])
        cu_b = torch.cat([cu[:1] + i * cap for i in range(b)]).contiguous()
        lens_b = torch.cat([lens[:1]] * b).contiguous()
        g = torch.Generator(device=dev).manual_seed(0xC0DE + b)
        q = torch.randn(b, L, wl.hq, wl.d, device=dev, generator=g).to(kf.dtype)
        kn = torch.randn(b, L, hkv, wl.d, device=dev, generator=g).to(kf.dtype)
        vn = torch.randn(b, L, hkv, wl.d, device=dev, generator=g).to(kf.dtype)
        out = torch.empty_like(q)
        wsb = torch.zeros(max(kv.kv_workspace_size(kv.KV_OP_DECODE, shape_b), 256),
                          dtype=torch.uint8, device=dev)
        scale = 1.0 / math.sqrt(wl.d)
        dts, byts = [], []
        for i in range(steps + 1):
            rows = int(lens_b.sum().item()) + b * L * hkv     # after this step's append
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            kv.flat_decode_attn(shape_b, q, kn, vn, kf_b, vf_b, cu_b, lens_b, scale, out, wsb,
                                stream)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            if i >= 1:
                dts.append(e0.elapsed_time(e1))
                byts.append(algorithmic_bytes(wl, b, L, 0, rows)["decode"])
        if kv.kv_check_device_status(wsb, stream):
            raise RuntimeError("device check in the batch-%d decode" % b)
        gbs = sum(byts) / (sum(dts) / 1e3) / 1e9
        res.append({"batch": b, "value": gbs, "unit": "GB/s", "steps": steps,
                    "ms_per_step": statistics.mean(dts), "bytes_per_step": statistics.mean(byts),
                    "cache": "%d replicas of sequence 0's flat cache at distinct addresses" % b})
        del kf_b, vf_b, q, kn, vn, out, wsb
        torch.cuda.empty_cache()
    return res


def decode_large(kv, W, dev, stream, flush, args):
    """flat_decode_attn alone on a flat cache of the batch-4, 32-layer, 32K-context
    Llama-3.1-8B-shaped set (1024 rows per KV head on average, log-normal spread, 256
    reserve rows), L2 flushed before each step."""
    import torch
    wl = W.WORKLOADS["llama8b_32k_b4"]
    fc = W.make_flat_cache(wl, mean_len=1024, sigma=0.7, reserve=256, seed=0xDEC0, device=dev)
    shape = kv.KvShape.from_workload(wl)
    wsd = torch.zeros(max(kv.kv_workspace_size(kv.KV_OP_DECODE, shape), 256), dtype=torch.uint8,
                      device=dev)
    out = torch.empty_like(fc["q"])
    scale = 1.0 / math.sqrt(wl.d)
    steps = 10
    B, L = wl.batch, wl.layers
    dts, byts = [], []
    for i in range(steps + 2):
        rows = int(fc["lens"].sum().item()) + B * L * wl.hkv     # after this step's append
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        kv.flat_decode_attn(shape, fc["q"], fc["k_new"], fc["v_new"], fc["k_flat"], fc["v_flat"],
                            fc["cu"], fc["lens"], scale, out, wsd, stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if i >= 2:
            dts.append(e0.elapsed_time(e1))
            byts.append(algorithmic_bytes(wl, B, L, 0, rows)["decode"])
    if kv.kv_check_device_status(wsd, stream):
        raise RuntimeError("device check in the large decode")
    gbs = sum(byts) / (sum(dts) / 1e3) / 1e9
    return {"value": gbs, "unit": "GB/s", "steps": steps,
            "ms_per_step": statistics.mean(dts), "bytes_per_step": statistics.mean(byts),
            "cache": "llama8b_32k_b4 shape: 1024 KV heads, 1024 rows each on average "
                     "(log-normal, sigma 0.7), 256 reserve rows; L2 flushed before each step"}


def time_crit_norm(kv, wl, shape, inp, crit, ws, dev, stream, reps=5):
    """crit_tc_kernel alone: kv_crit_norm (the CriticalKV norm by itself, one launch) between
    CUDA events on the launching stream, median of `reps` after one warm-up."""
    import torch
    B, L = shape.batch, shape.layers
    C = wl.n - wl.w
    ts = []
    for _ in range(reps + 1):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        kv.kv_crit_norm(shape, inp["v"], inp["w_o"], wl.model_dim, crit, ws, stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ts.append(e0.elapsed_time(e1))
    if kv.kv_check_device_status(ws, stream):
        raise RuntimeError("device check in kv_crit_norm")
    ms = statistics.median(ts[1:])
    flops = 2.0 * B * L * wl.hkv * C * wl.d * wl.model_dim
    tf = flops / (ms / 1e3) / 1e12
    tpeak, tkind = read_tensor_peak()
    return {"kernel": "crit_tc_kernel (||(V W_O)_j||_1 on tcgen05)", "ms": ms, "flops": flops,
            "achieved": tf, "unit": "TFLOP/s", "peak": tpeak, "frac": tf / tpeak,
            "peak_kind": tkind,
            "how": "kv_crit_norm alone between CUDA events, median of %d" % reps}


def time_call(fn, dev, stream, reps=3):
    """Median device time (ms) of fn() between CUDA events on `stream`, after one warm-up."""
    import torch
    ts = []
    for _ in range(reps + 1):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts[1:])


def measure_per_query_head(kv, wl, shape, inp, scores, dev, stream):
    """GQA-exact CriticalKV and LaProx on the workload's inputs, with one W_O block per query
    head ([L][Hq][d][D], N(0, 1/D)): per-query-head window terms (CUDA cores), the projected
    score on tcgen05 (2 * C * d * D flops per query head and unit, the dominant cost), then
    the selection each uses (two-stage with kappa given; model-wide TopK and per-head
    compaction).  Each call timed alone (median of 3)."""
    import torch
    B, L = shape.batch, shape.layers
    C = wl.n - wl.w
    D = wl.model_dim
    g = torch.Generator(device=dev).manual_seed(0x9A0)
    w_oq = (torch.randn(L, wl.hq, wl.d, D, device=dev, generator=g) / math.sqrt(D)).to(
        wl.torch_dtype)
    terms = torch.empty(B, L, wl.hq, C, device=dev)
    out = torch.empty(B, L, wl.hkv, C, device=dev)
    ws_s = torch.zeros(max(kv.kv_workspace_size(kv.KV_OP_SCORE, shape), 256), dtype=torch.uint8,
                       device=dev)
    ws_a = torch.zeros(max(kv.kv_workspace_size(kv.KV_OP_ALLOCATE, shape), 256),
                       dtype=torch.uint8, device=dev)
    ws_c = torch.zeros(max(kv.kv_workspace_size(kv.KV_OP_COMPACT, shape), 256), dtype=torch.uint8,
                       device=dev)
    tpeak, tkind = read_tensor_peak()
    flops = 2.0 * B * L * wl.hq * C * wl.d * D
    cap = wl.flat_capacity_rows()
    kept = torch.empty(cap, dtype=torch.int32, device=dev)
    cu = torch.empty(B, L, wl.hkv + 1, dtype=torch.int64, device=dev)
    lens = torch.empty(B, L, wl.hkv, dtype=torch.int32, device=dev)
    kf = torch.empty(cap, wl.d, dtype=wl.torch_dtype, device=dev)
    vf = torch.empty_like(kf)
    hb = torch.empty(B, L, wl.hkv, dtype=torch.int32, device=dev)
    lb = torch.empty(B, L, dtype=torch.int32, device=dev)
    budgets = wl.budgets().to(dev)
    res = {}
    for name, tk, pk in (("crit_gqa", kv.KV_TERMS_MEAN_POOLED, kv.KV_PROJ_CRIT_GQA),
                         ("laprox", kv.KV_TERMS_L2, kv.KV_PROJ_LAPROX)):
        t_terms = time_call(lambda: kv.kv_window_terms(shape, tk, inp["q_win"], inp["k"], terms,
                                                       ws_s, stream), dev, stream)
        t_proj = time_call(lambda: kv.kv_proj_score(shape, pk, inp["v"], w_oq, D, terms,
                                                    wl.crit_eps, out, ws_s, stream), dev, stream)
        tf = flops / (t_proj / 1e3) / 1e12
        r = {"terms_ms": t_terms, "proj_ms": t_proj, "proj_tflops": tf, "proj_frac": tf / tpeak,
             "peak_kind": tkind, "proj_flops": flops,
             "proj_kernel": "crit_tc_kernel, one W_O block per query head"}
        if name == "crit_gqa":
            kv.kv_allocate(shape, scores, budgets, 0, wl.alpha[0], wl.alpha[1], lb, hb, ws_a,
                           stream)
            r["select_ms"] = time_call(lambda: kv.kv_compact_kappa(
                shape, inp["k"], inp["v"], scores, out, wl.crit_alpha[0], wl.crit_alpha[1], hb,
                wl.reserve, kept, cu, lens, kf, vf, cap, ws_c, stream), dev, stream)
            r["select"] = "kv_compact_kappa (two-stage, kappa given)"
        else:
            total = torch.full((B,), int(budgets[0].sum().item()), dtype=torch.int64, device=dev)
            r["allocate_ms"] = time_call(lambda: kv.kv_allocate(
                shape, out, total, 2, 0, 1, lb, hb, ws_a, stream), dev, stream)
            r["select_ms"] = time_call(lambda: kv.kv_compact(
                shape, inp["k"], inp["v"], out, None, 1, 2, 0.0, hb, wl.reserve, kept, cu, lens,
                kf, vf, cap, ws_c, stream), dev, stream)
            r["allocate"] = "kv_allocate layer_entropy_mode 2 (model-wide TopK, %d layers)" % L
        for w_ in (ws_s, ws_a, ws_c):
            if kv.kv_check_device_status(w_, stream):
                raise RuntimeError("device check in the %s measurement" % name)
        res[name] = r
    del w_oq, terms, out, kf, vf, kept
    torch.cuda.empty_cache()
    return res


def measure_cascade_and_presets(kv, wl, shape, inp, scores, hb_main, flat, dev, stream):
    """The headline workload's other selection paths, timed alone on its inputs: LAVa's
    online prefill cascade (stage t: kv_allocate_capped over layers 0..t-1, kv_recompact of
    layers 0..t-2 from the previous flat cache, kv_recompact of layer t-1 from its K/V), the
    StreamingLLM preset (kv_compact_streaming), and the re-eviction of the flat cache after
    decode appends (kv_recompact); B = 1 for the cascade."""
    import torch
    B, L, hkv, n, w = shape.batch, shape.layers, wl.hkv, wl.n, wl.w
    total = wl.total_budget_value()
    reserve = wl.reserve
    cap = total + L * hkv * reserve
    flats = [{"kept": torch.empty(cap, dtype=torch.int32, device=dev),
              "cu": torch.zeros(1, L, hkv + 1, dtype=torch.int64, device=dev),
              "lens": torch.zeros(1, L, hkv, dtype=torch.int32, device=dev),
              "kf": torch.empty(cap, wl.d, dtype=wl.torch_dtype, device=dev),
              "vf": torch.empty(cap, wl.d, dtype=wl.torch_dtype, device=dev)} for _ in range(2)]
    caps = [torch.full((1, L), n * hkv, dtype=torch.int32, device=dev) for _ in range(2)]
    hbs = [torch.zeros(1, t, hkv, dtype=torch.int32, device=dev) for t in range(1, L + 1)]
    budget = torch.tensor([total], dtype=torch.int64, device=dev)
    sh = [kv.KvShape.from_workload(wl.with_(batch=1), layers=t) for t in range(0, L + 1)]
    w_a = torch.zeros(max(kv.kv_workspace_size(kv.KV_OP_ALLOCATE, shape), 256),
                      dtype=torch.uint8, device=dev)
    w_r = torch.zeros(kv.kv_recompact_workspace_size(max(cap, hkv * n)), dtype=torch.uint8,
                      device=dev)
    sc1 = scores[:1]
    k1, v1 = inp["k"][:1], inp["v"][:1]

    def cascade():
        for t in range(1, L + 1):
            lb, hb = caps[t % 2], hbs[t - 1]
            kv.kv_allocate_capped(sh[t], sc1[:, :t], budget, caps[(t - 1) % 2], 0, 1, lb, hb,
                                  w_a, stream)
            src, dst = flats[(t - 1) % 2], flats[t % 2]
            if t >= 2:
                kv.kv_recompact(sh[t - 1], sc1[:, :t - 1], hb[:, :t - 1], src["kept"],
                                src["cu"][:, :t - 1], src["lens"][:, :t - 1], src["kf"],
                                src["vf"], reserve, None, dst["kept"], dst["cu"], dst["lens"],
                                dst["kf"], dst["vf"], w_r, stream)
            row_base = dst["cu"][0, t - 2, hkv:hkv + 1] if t >= 2 else None
            kv.kv_recompact(sh[1], sc1[:, t - 1:t], hb[:, t - 1:t], None, None, None,
                            k1[:, t - 1:t], v1[:, t - 1:t], reserve, row_base, dst["kept"],
                            dst["cu"][:, t - 1:t], dst["lens"][:, t - 1:t], dst["kf"], dst["vf"],
                            w_r, stream)

    # the slices above must be contiguous views (B = 1, or the first sequence)
    t_cascade = time_call(cascade, dev, stream, reps=2)
    for w_ in (w_a, w_r):
        if kv.kv_check_device_status(w_, stream):
            raise RuntimeError("device check in the cascade measurement")
    rows_final = int(flats[L % 2]["lens"].sum().item())
    peak_rows = total + n * hkv
    res = {"cascade": {"ms": t_cascade, "stages": L, "ms_per_stage": t_cascade / L,
                       "rows_final": rows_final, "peak_rows": peak_rows,
                       "peak_rows_one_shot": L * n * hkv,
                       "how": "32 stages of kv_allocate_capped + 2 kv_recompact, eager"}}
    del flats
    torch.cuda.empty_cache()
    # StreamingLLM preset with the workload's own per-head budgets
    row_bytes = wl.d * wl.elem_bytes
    capm = wl.flat_capacity_rows()
    out = {k_: torch.empty_like(x) for k_, x in flat.items()}
    ws1 = torch.zeros(256, dtype=torch.uint8, device=dev)
    t_st = time_call(lambda: kv.kv_compact_streaming(
        shape, inp["k"], inp["v"], 4, hb_main, reserve, out["kept"], out["cu"], out["lens"],
        out["kf"], out["vf"], capm, ws1, stream), dev, stream)
    rows = int(hb_main.sum().item())
    st_bytes = 4 * rows * row_bytes + 4 * rows
    res["streaming"] = {"ms": t_st, "rows": rows, "gbs": st_bytes / (t_st / 1e3) / 1e9,
                        "how": "kv_compact_streaming (4 sinks), the workload's head budgets"}
    # re-eviction of the decoded flat cache: every head up to 16 prefill rows smaller (its
    # window and appended rows stay)
    new_hb = (flat["lens"] - torch.clamp(hb_main - wl.w, max=16)).to(torch.int32)
    ws_r = torch.zeros(kv.kv_recompact_workspace_size(capm), dtype=torch.uint8, device=dev)
    t_re = time_call(lambda: kv.kv_recompact(
        shape, scores, new_hb, flat["kept"], flat["cu"], flat["lens"], flat["kf"], flat["vf"],
        reserve, None, out["kept"], out["cu"], out["lens"], out["kf"], out["vf"], ws_r, stream),
        dev, stream)
    rows = int(new_hb.sum().item())
    re_bytes = 4 * rows * row_bytes + 8 * rows + 4 * int(flat["lens"].sum().item())
    res["reevict"] = {"ms": t_re, "rows": rows, "gbs": re_bytes / (t_re / 1e3) / 1e9,
                      "how": "kv_recompact of the decoded flat cache, 16 prefill rows fewer "
                             "per head (appended and window rows kept)"}
    for w_ in (ws1, ws_r):
        if kv.kv_check_device_status(w_, stream):
            raise RuntimeError("device check in the preset measurements")
    del out
    torch.cuda.empty_cache()
    return res


def measure_workload(kv, W, wl, dev, stream, steps, warmup):
    """One more workload of the pages' configurations: the same step as the headline (eviction
    pass over every (sequence, layer), then one decode step over every layer), eager launches
    with CUDA events between the stages, inputs resident in HBM (larger than L2 except for
    the one-layer workload, which flushes L2 between steps).  Its tensors are freed on
    return."""
    import torch
    B, L = wl.batch, wl.layers
    C = wl.n - wl.w
    shape = kv.KvShape.from_workload(wl)
    mode = {"ada": kv.KV_SCORE_ADA, "lava": kv.KV_SCORE_LAVA, "critical": kv.KV_SCORE_CRITICAL}[
        wl.mode]
    group = kv.KV_GROUP_MAX if wl.group == "max" else kv.KV_GROUP_MEAN
    entropy = 1 if wl.budget_kind == "total" else 0
    inp = W.make_batch(wl, device=dev)
    budgets = wl.budgets().to(dev)
    dec = W.make_decode_batch(wl, 0, inp["tau"], device=dev)
    cap = wl.flat_capacity_rows()

    def ws(op):
        return torch.zeros(max(kv.kv_workspace_size(op, shape), 256), dtype=torch.uint8,
                           device=dev)

    w_s, w_a, w_c, w_d = (ws(kv.KV_OP_SCORE), ws(kv.KV_OP_ALLOCATE), ws(kv.KV_OP_COMPACT),
                          ws(kv.KV_OP_DECODE))
    scores = torch.empty(B, L, wl.hkv, C, dtype=torch.float32, device=dev)
    crit = torch.empty_like(scores) if wl.mode == "critical" else None
    lb = torch.empty(B, L, dtype=torch.int32, device=dev)
    hb = torch.empty(B, L, wl.hkv, dtype=torch.int32, device=dev)
    kept = torch.empty(cap, dtype=torch.int32, device=dev)
    cu = torch.empty(B, L, wl.hkv + 1, dtype=torch.int64, device=dev)
    lens = torch.empty(B, L, wl.hkv, dtype=torch.int32, device=dev)
    kf = torch.empty(cap, wl.d, dtype=wl.torch_dtype, device=dev)
    vf = torch.empty_like(kf)
    out = torch.empty_like(dec["q"])
    scale = 1.0 / math.sqrt(wl.d)
    input_bytes = 2 * inp["k"].numel() * inp["k"].element_size()
    flush = (torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
             if input_bytes <= 2 * L2_BYTES else None)

    def step(ev):
        ev[0].record(stream)
        kv.kv_score(shape, mode, group, inp["q_win"], inp["k"],
                    inp["v"] if wl.mode != "ada" else None, inp["w_o"], wl.model_dim, scores,
                    crit, w_s, stream)
        ev[1].record(stream)
        kv.kv_allocate(shape, scores, budgets, entropy, wl.alpha[0], wl.alpha[1], lb, hb, w_a,
                       stream)
        ev[2].record(stream)
        kv.kv_compact(shape, inp["k"], inp["v"], scores, crit, wl.crit_alpha[0],
                      wl.crit_alpha[1], wl.crit_eps, hb, wl.reserve, kept, cu, lens, kf, vf, cap,
                      w_c, stream)
        ev[3].record(stream)
        kv.flat_decode_attn(shape, dec["q"], dec["k_new"], dec["v_new"], kf, vf, cu, lens, scale,
                            out, w_d, stream)
        ev[4].record(stream)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)]
           for _ in range(warmup + steps)]
    for i in range(warmup + steps):
        if flush is not None:
            flush.zero_()
        step(evs[i])
    torch.cuda.synchronize(dev)
    for w_ in (w_s, w_a, w_c, w_d):
        if kv.kv_check_device_status(w_, stream):
            raise RuntimeError("device check in the %s step" % wl.name)
    timed = evs[warmup:]
    names = ["score", "allocate", "compact", "decode"]
    stages = {nm: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in timed)
              for j, nm in enumerate(names)}
    ms = statistics.mean(e[0].elapsed_time(e[4]) for e in timed)
    t_evict = stages["score"] + stages["allocate"] + stages["compact"]
    hb_rows = int(hb.sum().item())
    rows = int(lens.sum().item())
    ab = algorithmic_bytes(wl, B, L, hb_rows, rows)
    peak = read_peaks()[0]
    res = {"workload": wl.name, "batch": B, "layers": L, "n": wl.n, "score": wl.mode,
           "budget": ("total %d per sequence" % wl.total_budget_value()
                      if wl.budget_kind == "total" else
                      "%d per layer" % wl.layer_budget_value()),
           "ms_per_step": ms, "value": aggregate_value(1, B, wl.n, L, ms), "unit": UNIT,
           "eviction_only": aggregate_value(1, B, wl.n, L, t_evict), "stages_ms": stages,
           "score_gbs": ab["score"] / (stages["score"] / 1e3) / 1e9,
           "eviction_frac_of_hbm": (ab["score"] + ab["allocate"] + ab["compact"]) /
           (t_evict / 1e3) / 1e9 / peak,
           "decode_gbs_in_step": ab["decode"] / (stages["decode"] / 1e3) / 1e9,
           "steps": steps, "timing": "eager launches, CUDA events between the stages",
           "l2": "flushed before each step" if flush is not None else
           "inputs larger than L2 (K+V %.1f GiB)" % (input_bytes / 2**30)}
    if wl.mode == "critical":
        res["crit_norm"] = time_crit_norm(kv, wl, shape, inp, crit, w_s, dev, stream)
        res["per_query_head"] = measure_per_query_head(kv, wl, shape, inp, scores, dev, stream)
    del inp, scores, crit, kf, vf, kept, flush
    torch.cuda.empty_cache()
    return res


# Workloads timed after the headline one on the default run: the pages' other
# configurations (the one-layer 16K sweep at three budgets, the 4 x 32-layer 32K set and the
# 32-layer 64K CriticalKV set).
OTHER_WORKLOADS = (("llama8b_16k_layer", {"head_budget_frac": 0.2}),
                   ("llama8b_16k_layer", {"head_budget_frac": 0.4}),
                   ("llama8b_16k_layer", {"head_budget_frac": 0.8}),
                   ("llama8b_32k_b4", {}),
                   ("llama8b_64k_criticalkv", {}))


def run_decode_only(args, kv, W, dev):
    """flat_decode_attn alone, L2 flushed before each step, on a flat cache of the workload's
    shape whose head lengths are log-normal (--decode-sigma) around the workload's mean rows
    per head: the decode of the eviction pass's output without its inputs on the device."""
    import torch
    wl = W.WORKLOADS[args.workload]
    if args.layers > 0:
        wl = wl.with_(layers=args.layers)
    if wl.budget_kind == "total":
        mean = wl.total_per_head_layer
    else:
        mean = wl.layer_budget_value() // wl.hkv
    reserve = max(wl.reserve, 8)
    fc = W.make_flat_cache(wl, mean_len=mean, sigma=args.decode_sigma, reserve=reserve,
                           seed=0xDEC1, device=dev)
    shape = kv.KvShape.from_workload(wl)
    wsd = torch.zeros(max(kv.kv_workspace_size(kv.KV_OP_DECODE, shape), 256), dtype=torch.uint8,
                      device=dev)
    out = torch.empty_like(fc["q"])
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    scale = 1.0 / math.sqrt(wl.d)
    B, L = wl.batch, wl.layers
    steps = max(1, min(args.decode_steps if args.decode_steps > 0 else 32, reserve - 1))
    dts, byts = [], []
    for i in range(max(args.warmup, 0) + steps):
        rows = int(fc["lens"].sum().item()) + B * L * wl.hkv
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        kv.flat_decode_attn(shape, fc["q"], fc["k_new"], fc["v_new"], fc["k_flat"], fc["v_flat"],
                            fc["cu"], fc["lens"], scale, out, wsd, stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if i >= max(args.warmup, 0):
            dts.append(e0.elapsed_time(e1))
            byts.append(algorithmic_bytes(wl, B, L, 0, rows)["decode"])
    if kv.kv_check_device_status(wsd, stream):
        raise RuntimeError("device check in the decode-only run")
    peak, peak_kind = read_peaks()
    gbs = sum(byts) / (sum(dts) / 1e3) / 1e9
    print(json.dumps({
        "metric": "flat varlen decode attn HBM GB/s", "value": gbs, "unit": "GB/s",
        "frac": gbs / peak, "peak": peak, "peak_kind": peak_kind, "n_gpus": 1, "steps": steps,
        "warmup": args.warmup, "ms_per_step": statistics.mean(dts),
        "bytes_per_step": statistics.mean(byts), "higher_is_better": True,
        "data": "synthetic flat cache (log-normal head lengths, sigma %g, around %d rows, "
                "longest %d)" % (args.decode_sigma, mean, int(fc["lens"].max().item())),
        "config": {"workload": wl.name, "batch": B, "layers": L, "hkv": wl.hkv, "hq": wl.hq,
                   "d": wl.d, "reserve": reserve, "l2": "flushed before each step"}}),
          flush=True)
    return 0


def run_ours(args):
    import torch
    import kv_cache_eviction_gb300 as kv
    from kv_cache_eviction_gb300 import workloads as W
    import __graft_entry__

    rank, world, local = dist_env()
    wl = W.WORKLOADS[args.workload]
    if args.layers > 0:
        wl = wl.with_(layers=args.layers)
    # the CPU oracle first: its process pool is forked before this process touches the GPU
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.decode_only:
        cpu = cpu_baseline(wl)
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.decode_only:
        if rank != 0:
            return 0
        __graft_entry__.build()
        return run_decode_only(args, kv, W, dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    __graft_entry__.build()

    B, L = wl.batch, wl.layers
    seqs = rank_sequences(rank, B)
    shape = kv.KvShape.from_workload(wl)
    C = wl.n - wl.w
    mode = {"ada": kv.KV_SCORE_ADA, "lava": kv.KV_SCORE_LAVA, "critical": kv.KV_SCORE_CRITICAL}[
        wl.mode]
    group = kv.KV_GROUP_MAX if wl.group == "max" else kv.KV_GROUP_MEAN
    entropy = 1 if wl.budget_kind == "total" else 0

    inp = W.make_batch(wl, device=dev, seqs=seqs)
    budgets = wl.budgets().to(dev)
    dec = W.make_decode_batch(wl, 0, inp["tau"], device=dev, seqs=seqs)
    cap = wl.flat_capacity_rows()

    def ws(op):
        return torch.zeros(max(kv.kv_workspace_size(op, shape), 256), dtype=torch.uint8,
                           device=dev)

    w_s, w_a, w_c, w_d = (ws(kv.KV_OP_SCORE), ws(kv.KV_OP_ALLOCATE), ws(kv.KV_OP_COMPACT),
                          ws(kv.KV_OP_DECODE))
    scores = torch.empty(B, L, wl.hkv, C, dtype=torch.float32, device=dev)
    crit = torch.empty_like(scores) if wl.mode == "critical" else None
    lb = torch.empty(B, L, dtype=torch.int32, device=dev)
    hb = torch.empty(B, L, wl.hkv, dtype=torch.int32, device=dev)
    kept = torch.empty(cap, dtype=torch.int32, device=dev)
    cu = torch.empty(B, L, wl.hkv + 1, dtype=torch.int64, device=dev)
    lens = torch.empty(B, L, wl.hkv, dtype=torch.int32, device=dev)
    kf = torch.empty(cap, wl.d, dtype=wl.torch_dtype, device=dev)
    vf = torch.empty_like(kf)
    out = torch.empty_like(dec["q"])
    scale = 1.0 / math.sqrt(wl.d)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def step(ev=None, st=None, score=True):
        st = stream if st is None else st
        if ev is not None:
            ev[0].record(st)
        if score:
            kv.kv_score(shape, mode, group, inp["q_win"], inp["k"],
                        inp["v"] if wl.mode != "ada" else None, inp["w_o"], wl.model_dim,
                        scores, crit, w_s, st)
        if ev is not None:
            ev[1].record(st)
        kv.kv_allocate(shape, scores, budgets, entropy, wl.alpha[0], wl.alpha[1], lb, hb, w_a,
                       st)
        if ev is not None:
            ev[2].record(st)
        kv.kv_compact(shape, inp["k"], inp["v"], scores, crit, wl.crit_alpha[0],
                      wl.crit_alpha[1], wl.crit_eps, hb, wl.reserve, kept, cu, lens, kf, vf, cap,
                      w_c, st)
        if ev is not None:
            ev[3].record(st)
        kv.flat_decode_attn(shape, dec["q"], dec["k_new"], dec["v_new"], kf, vf, cu, lens, scale,
                            out, w_d, st)
        if ev is not None:
            ev[4].record(st)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(max(args.warmup, 0)):
        step()
    torch.cuda.synchronize(dev)
    for w_ in (w_s, w_a, w_c, w_d):
        code = kv.kv_check_device_status(w_, stream)
        if code:
            raise RuntimeError("device check %d during warm-up" % code)

    input_bytes = 2 * inp["k"].numel() * inp["k"].element_size()
    big_inputs = input_bytes > 2 * L2_BYTES
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local) if rank == 0 else None
    launches0 = kv.kv_kernel_launches()
    barrier()
    torch.cuda.synchronize(dev)
    t_start.record(stream)
    for i in range(args.steps):
        if not big_inputs and i > 0:
            flush.zero_()
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    launches = kv.kv_kernel_launches() - launches0

    stage_names = ["score", "allocate", "compact", "decode"]
    stage_ms = {nm: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1])
                                    for i in range(args.steps))
                for j, nm in enumerate(stage_names)}
    if big_inputs:
        eager_ms = t_start.elapsed_time(t_end) / args.steps
    else:
        eager_ms = statistics.mean(evs[i][0].elapsed_time(evs[i][4])
                                   for i in range(args.steps))
    for w_ in (w_s, w_a, w_c, w_d):
        code = kv.kv_check_device_status(w_, stream)
        if code:
            raise RuntimeError("device check %d in the timed region" % code)

    # -------------------- the same step captured once as a CUDA graph --------------------
    # The four calls enqueue every kernel on one stream with no host work between them, so
    # the step can be captured and replayed: one graph launch per step instead of the
    # library's host-side launches.  Only with inputs larger than L2 (no flush to interleave).
    graph_ms, graph_note = None, None
    if args.no_graph:
        graph_note = "not run (--no-graph)"
    elif not big_inputs:
        graph_note = "not run (inputs fit in L2: the flush between steps is not in the graph)"
    else:
        try:
            gs = torch.cuda.Stream(dev)
            gs.wait_stream(stream)
            torch.cuda.synchronize(dev)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=gs):
                step(st=gs)
            with torch.cuda.stream(gs):
                for _ in range(max(args.warmup, 0)):
                    graph.replay()
                torch.cuda.synchronize(dev)
                g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                barrier()
                torch.cuda.synchronize(dev)
                g0.record(gs)
                for _ in range(args.steps):
                    graph.replay()
                g1.record(gs)
                torch.cuda.synchronize(dev)
            barrier()
            graph_ms = g0.elapsed_time(g1) / args.steps
            for w_ in (w_s, w_a, w_c, w_d):
                code = kv.kv_check_device_status(w_, stream)
                if code:
                    raise RuntimeError("device check %d in the graph replays" % code)
            graph_note = "one CUDA graph per step (captured once), replayed %d times" % args.steps
            del graph
        except RuntimeError as e:
            if "device check" in str(e):
                raise
            graph_note = "capture failed: " + str(e).splitlines()[0][:160]
            graph_ms = None
            torch.cuda.synchronize(dev)
    clk = clocks.stop() if clocks is not None else None
    ms_per_step = graph_ms if graph_ms is not None else eager_ms
    t_local = max_over_ranks(ms_per_step, dev)
    value = aggregate_value(world, B, wl.n, L, t_local)

    # -------------------- decode alone, L2 flushed before each step --------------------
    hb_rows = int(hb.sum().item())
    lens0 = int(lens.sum().item())          # includes the timed region's last append
    nd = wl.decode_steps if args.decode_steps < 0 else args.decode_steps
    nd = max(1, min(nd, wl.reserve - 1))
    # rebuild the flat cache so every decode step has a reserve row
    kv.kv_compact(shape, inp["k"], inp["v"], scores, crit, wl.crit_alpha[0], wl.crit_alpha[1],
                  wl.crit_eps, hb, wl.reserve, kept, cu, lens, kf, vf, cap, w_c, stream)
    lens0 = int(lens.sum().item())
    # Even steps launch eagerly, odd steps replay one captured CUDA graph of the call (what a
    # serving loop does) with the step's inputs copied into the captured buffers first: both
    # see the same growing cache.  Both are reported; the graph time is the value when the
    # capture works.
    d0 = W.make_decode_batch(wl, 1, inp["tau"], device=dev, seqs=seqs)
    xq, xk, xv = d0["q"].clone(), d0["k_new"].clone(), d0["v_new"].clone()
    dec_t = {"eager": ([], []), "graph": ([], [])}   # times, bytes
    dec_graph, dec_note = None, "not run (--no-graph)" if args.no_graph else None
    gsd = torch.cuda.Stream(dev)
    if not args.no_graph and nd >= 2:
        gsd.wait_stream(stream)
        torch.cuda.synchronize(dev)
        try:
            dec_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(dec_graph, stream=gsd):
                kv.flat_decode_attn(shape, xq, xk, xv, kf, vf, cu, lens, scale, out, w_d, gsd)
        except RuntimeError as e:
            dec_graph, dec_note = None, "capture failed: " + str(e).splitlines()[0][:160]
            torch.cuda.synchronize(dev)
    for s_ in range(nd):
        d_in = W.make_decode_batch(wl, 1 + s_, inp["tau"], device=dev, seqs=seqs)
        kind = "graph" if dec_graph is not None and s_ % 2 == 1 else "eager"
        st_ = gsd if kind == "graph" else stream
        with torch.cuda.stream(st_):
            if kind == "graph":
                xq.copy_(d_in["q"])
                xk.copy_(d_in["k_new"])
                xv.copy_(d_in["v_new"])
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st_)
            if kind == "graph":
                dec_graph.replay()
            else:
                kv.flat_decode_attn(shape, d_in["q"], d_in["k_new"], d_in["v_new"], kf, vf, cu,
                                    lens, scale, out, w_d, st_)
            e1.record(st_)
        torch.cuda.synchronize(dev)
        rows = lens0 + (s_ + 1) * B * L * wl.hkv
        dec_t[kind][0].append(e0.elapsed_time(e1))
        dec_t[kind][1].append(algorithmic_bytes(wl, B, L, hb_rows, rows)["decode"])
    if kv.kv_check_device_status(w_d, stream):
        raise RuntimeError("device check in decode")
    del dec_graph
    peak, peak_kind = read_peaks()
    dec_kind = "graph" if dec_t["graph"][0] else "eager"
    dts, dbytes = dec_t[dec_kind]
    dec_eager_gbs = (sum(dec_t["eager"][1]) / (sum(dec_t["eager"][0]) / 1e3) / 1e9
                     if dec_t["eager"][0] else None)
    dec_gbs = sum(dbytes) / (sum(dts) / 1e3) / 1e9

    # -------------------- decode alone, one launch per layer --------------------
    # The serving loop's own shape: each layer's decode is its own call (one sequence, the
    # layer's Hkv heads).  The L calls of a step are captured once as a CUDA graph and
    # replayed (a launch loop in Python would time the host, not the GPU), with the step's
    # inputs copied into the captured buffers and L2 flushed before each replay.
    dec_pl = None
    if B == 1 and L > 1 and not args.no_decode_per_layer:
        shape1 = kv.KvShape.from_workload(wl.with_(layers=1))
        w_d1 = torch.zeros(max(kv.kv_workspace_size(kv.KV_OP_DECODE, shape1), 256),
                           dtype=torch.uint8, device=dev)
        kv.kv_compact(shape, inp["k"], inp["v"], scores, crit, wl.crit_alpha[0], wl.crit_alpha[1],
                      wl.crit_eps, hb, wl.reserve, kept, cu, lens, kf, vf, cap, w_c, stream)
        # per-layer offset tables on 16-byte boundaries (the ABI's alignment rule)
        cu_pl = torch.zeros(L, 16, dtype=torch.int64, device=dev)
        cu_pl[:, :wl.hkv + 1] = cu[0]
        d0 = W.make_decode_batch(wl, 1, inp["tau"], device=dev, seqs=seqs)
        xq, xk, xv = d0["q"].clone(), d0["k_new"].clone(), d0["v_new"].clone()

        def layer_calls(st):
            for l in range(L):
                kv.flat_decode_attn(shape1, xq[0, l], xk[0, l], xv[0, l], kf, vf, cu_pl[l],
                                    lens[0, l], scale, out[0, l], w_d1, st,
                                    flat_capacity_rows=cap)

        gs = torch.cuda.Stream(dev)
        gs.wait_stream(stream)
        torch.cuda.synchronize(dev)
        pl_graph, pl_note = None, None
        try:
            pl_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(pl_graph, stream=gs):
                layer_calls(gs)
        except RuntimeError as e:
            pl_graph, pl_note = None, "capture failed: " + str(e).splitlines()[0][:160]
            torch.cuda.synchronize(dev)
        lens_pl0 = int(lens.sum().item())
        pl = {"graph": ([], []), "eager": ([], [])}   # times, bytes
        with torch.cuda.stream(gs):
            for s_ in range(nd):
                d_in = W.make_decode_batch(wl, 1 + s_, inp["tau"], device=dev, seqs=seqs)
                xq.copy_(d_in["q"])
                xk.copy_(d_in["k_new"])
                xv.copy_(d_in["v_new"])
                flush.zero_()
                # the last step (or every step without a graph) launches eagerly
                kind = "graph" if pl_graph is not None and s_ < nd - 1 else "eager"
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(gs)
                if kind == "graph":
                    pl_graph.replay()
                else:
                    layer_calls(gs)
                e1.record(gs)
                torch.cuda.synchronize(dev)
                rows = lens_pl0 + (s_ + 1) * L * wl.hkv
                pl[kind][0].append(e0.elapsed_time(e1))
                pl[kind][1].append(algorithmic_bytes(wl, B, L, hb_rows, rows)["decode"])
        if kv.kv_check_device_status(w_d1, stream):
            raise RuntimeError("device check in the per-layer decode")
        kind = "graph" if pl["graph"][0] else "eager"
        timed, tbytes = pl[kind]
        pl_gbs = sum(tbytes) / (sum(timed) / 1e3) / 1e9
        dec_pl = {"value": pl_gbs, "unit": "GB/s", "frac": pl_gbs / peak, "steps": len(timed),
                  "ms_per_step": statistics.mean(timed), "launches_per_step": L,
                  "timing": ("CUDA graph of the %d per-layer calls, replayed" % L)
                  if kind == "graph" else "eager per-layer calls (graph: %s)" % pl_note,
                  "eager_us_per_call": statistics.mean(pl["eager"][0]) * 1e3 / L
                  if pl["eager"][0] else None,
                  "l2": "flushed before each step of %d per-layer calls" % L}
        del pl_graph
    dec_batches = None
    if args.decode_batches and rank == 0:
        kv.kv_compact(shape, inp["k"], inp["v"], scores, crit, wl.crit_alpha[0],
                      wl.crit_alpha[1], wl.crit_eps, hb, wl.reserve, kept, cu, lens, kf, vf, cap,
                      w_c, stream)
        dec_batches = decode_batches(kv, W, wl, dev, stream, flush, kf, vf, cu, lens, cap,
                                     [int(x) for x in args.decode_batches.split(",") if x])
        peak_ = read_peaks()[0]
        for r in dec_batches:
            r["frac"] = r["value"] / peak_
    dec_large = (decode_large(kv, W, dev, stream, flush, args)
                 if rank == 0 and not args.no_decode_large else None)

    # -------------------- roofline of the dominant stage --------------------
    ab = algorithmic_bytes(wl, B, L, hb_rows, lens0)
    dom = max(("score", "allocate", "compact"), key=lambda k: stage_ms[k])
    achieved = ab[dom] / (stage_ms[dom] / 1e3) / 1e9
    roofline = {"kernel": "kv_score (window scoring)" if dom == "score" else dom,
                "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_kind": peak_kind,
                "traffic": read_traffic(wl.name) if dom == "score" else None,
                "algorithmic_bytes_per_launch": ab[dom]}
    crit_norm = None
    if wl.mode == "critical":
        crit_norm = time_crit_norm(kv, wl, shape, inp, crit, w_s, dev, stream)
        roofline = {"kernel": crit_norm["kernel"], "bound": "tensor",
                    "achieved": crit_norm["achieved"], "peak": crit_norm["peak"],
                    "unit": "TFLOP/s", "frac": crit_norm["frac"],
                    "peak_kind": crit_norm["peak_kind"], "traffic": None,
                    "flops_per_launch": crit_norm["flops"], "how": crit_norm["how"]}

    # -------------------- end to end through host buffers --------------------
    e2e = None
    if args.e2e_steps > 0:
        # The inputs sit in page-locked host buffers backed by huge pages (the package's
        # pinned_empty): copies from torch's pinned memory on this host's 64 KB pages ran at
        # 28-211 GB/s from one copy to the next, from huge-page buffers at 211 GB/s.
        from kv_cache_eviction_gb300.hostmem import pinned_empty
        host = {}
        h2d = 0
        for name in ("q_win", "k", "v", "w_o"):
            t = inp.get(name)
            if t is None or (name == "v" and wl.mode == "ada"):
                continue
            host[name] = pinned_empty(t.shape, t.dtype)
            host[name].copy_(t)
            h2d += t.numel() * t.element_size()
        for name in ("q", "k_new", "v_new"):
            host["dec_" + name] = pinned_empty(dec[name].shape, dec[name].dtype)
            host["dec_" + name].copy_(dec[name])
            h2d += dec[name].numel() * dec[name].element_size()
        budgets_h = budgets.cpu().pin_memory()
        h2d += budgets.numel() * budgets.element_size()
        res = {"out": torch.empty(out.shape, dtype=out.dtype, pin_memory=True),
               "hb": torch.empty(hb.shape, dtype=hb.dtype, pin_memory=True),
               "lb": torch.empty(lb.shape, dtype=lb.dtype, pin_memory=True),
               "lens": torch.empty(lens.shape, dtype=lens.dtype, pin_memory=True)}
        d2h = sum(t.numel() * t.element_size() for t in res.values())
        # The copies are bound by the host link (211 GB/s here, for copy engines and SM loads
        # alike), so the scoring overlaps them: the layers go over in chunks on a copy
        # stream, and each chunk is scored as soon as it is on the device.  Allocation (whose
        # layer budgets need every layer), compaction and the decode step follow the last.
        nch = 8 if (B == 1 and L % 8 == 0) else 1
        Lc = L // nch
        shape_c = kv.KvShape.from_workload(wl.with_(layers=Lc)) if nch > 1 else shape
        cstream = torch.cuda.Stream(dev)

        def layer_slice(name, t, l0, l1):
            return t[l0:l1] if name == "w_o" else t[:, l0:l1]

        e2e_ms = []
        for it in range(args.e2e_steps + 1):     # the first pass is untimed (warm-up)
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            cstream.wait_event(e0)
            chunk_ev = [torch.cuda.Event() for _ in range(nch + 1)]
            with torch.cuda.stream(cstream):
                for c in range(nch):
                    l0, l1 = c * Lc, (c + 1) * Lc
                    for name in ("q_win", "k", "v", "w_o"):
                        if name in host:
                            layer_slice(name, inp[name], l0, l1).copy_(
                                layer_slice(name, host[name], l0, l1), non_blocking=True)
                    chunk_ev[c].record(cstream)
                for name in ("q", "k_new", "v_new"):
                    dec[name].copy_(host["dec_" + name], non_blocking=True)
                budgets.copy_(budgets_h, non_blocking=True)
                chunk_ev[nch].record(cstream)
            if nch > 1:
                for c in range(nch):
                    l0, l1 = c * Lc, (c + 1) * Lc
                    stream.wait_event(chunk_ev[c])
                    kv.kv_score(shape_c, mode, group, inp["q_win"][:, l0:l1], inp["k"][:, l0:l1],
                                inp["v"][:, l0:l1] if wl.mode != "ada" else None,
                                inp["w_o"][l0:l1] if inp.get("w_o") is not None else None,
                                wl.model_dim, scores[:, l0:l1],
                                crit[:, l0:l1] if crit is not None else None, w_s, stream)
                stream.wait_event(chunk_ev[nch])
                step(score=False)
            else:
                stream.wait_event(chunk_ev[nch])
                step()
            res["out"].copy_(out, non_blocking=True)
            res["hb"].copy_(hb, non_blocking=True)
            res["lb"].copy_(lb, non_blocking=True)
            res["lens"].copy_(lens, non_blocking=True)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            if it > 0:
                e2e_ms.append(e0.elapsed_time(e1))
        t_e2e = max_over_ranks(statistics.median(e2e_ms), dev)
        e2e = {"value": aggregate_value(world, B, wl.n, L, t_e2e), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e,
               "steps": args.e2e_steps,
               "how": ("inputs (page-locked huge-page host buffers) copied in %d layer chunks on "
                       "a copy stream, each chunk scored as it lands" % nch) if nch > 1 else
                      "inputs (page-locked huge-page host buffers) copied, then the step"}
        del host

    # -------------------- the headline workload's other selection paths --------------------
    paths = None
    if (rank == 0 and world == 1 and not args.no_other_workloads and args.layers <= 0 and
            wl.mode == "lava" and B == 1):
        paths = measure_cascade_and_presets(
            kv, wl, shape, inp, scores, hb,
            {"kept": kept, "cu": cu, "lens": lens, "kf": kf, "vf": vf}, dev, stream)

    # -------------------- the pages' other configurations --------------------
    others = None
    if rank == 0 and world == 1 and not args.no_other_workloads and args.layers <= 0:
        del step, inp, dec, scores, crit, kept, kf, vf, out, flush
        torch.cuda.empty_cache()
        others = []
        for name, kw in OTHER_WORKLOADS:
            if name == wl.name and not kw:
                continue
            others.append(measure_workload(kv, W, W.WORKLOADS[name].with_(**kw), dev, stream,
                                           steps=min(args.steps, 10), warmup=3))
    t_evict = stage_ms["score"] + stage_ms["allocate"] + stage_ms["compact"]

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
            if wl.dtype == "bf16" else "f32",
            "data": "synthetic (seeded generator; shapes of the pages' workloads)",
            "config": {
                "workload": wl.name, "batch_per_gpu": B, "layers": L, "hq": wl.hq,
                "hkv": wl.hkv, "d": wl.d, "n": wl.n, "w": wl.w, "pool": wl.pool,
                "score": wl.mode, "group": wl.group,
                "budget": ("total %d per sequence" % wl.total_budget_value()
                           if wl.budget_kind == "total" else
                           "%d per layer" % wl.layer_budget_value()),
                "alpha": "%d/%d" % wl.alpha, "accumulate": "f32",
                "parallelism": "replicas (independent sequences per GPU)" if world > 1 else
                "1 GPU",
                "l2": ("inputs larger than L2 (K+V %.1f GiB per step)" % (input_bytes / 2**30))
                if big_inputs else "L2 flushed between steps",
                "step": "kv_score + kv_allocate + kv_compact over all layers, then one "
                        "flat_decode_attn step over all layers",
                "timing": graph_note if graph_ms is not None else
                "eager launches (graph: %s)" % graph_note,
            },
            "eager_ms_per_step": eager_ms,
            "stages_ms": stage_ms,
            "eviction_only": {"value": aggregate_value(world, B, wl.n, L, t_evict),
                              "unit": UNIT, "ms": t_evict,
                              "how": "score + allocate + compact stage times (eager)"},
            "decode_attn": {"value": dec_gbs, "unit": "GB/s", "frac": dec_gbs / peak,
                            "peak": peak, "steps": len(dts), "ms_per_step": statistics.mean(dts),
                            "bytes_per_step": statistics.mean(dbytes),
                            "timing": "one captured CUDA graph of the call, replayed"
                            if dec_kind == "graph" else
                            "eager launches (graph: %s)" % (dec_note or "not run"),
                            "eager_value": dec_eager_gbs,
                            "eager_ms_per_step": statistics.mean(dec_t["eager"][0])
                            if dec_t["eager"][0] else None,
                            "l2": "flushed before each step"},
            "decode_attn_per_layer": dec_pl,
            "decode_attn_batches": dec_batches,
            "decode_attn_large": dict(dec_large, frac=dec_large["value"] / peak)
            if dec_large else None,
            "roofline": roofline,
            "crit_norm": crit_norm,
            "cpu_baseline": cpu,
            "workloads": others,
            "selection_paths": paths,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
