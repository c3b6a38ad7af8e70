"""The bench's multi-rank logic with two gloo ranks on CPU.

`bench.py --gpus N` runs one process per GPU; each evicts its own sequences (no data-path
exchange), the step time is the slowest rank's, and the value aggregates every rank's
tokens.  These tests run that logic as two real processes over gloo.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from kv_cache_eviction_gb300 import workloads as W
        t_local = 2.0 + 0.75 * rank                    # ms: rank 1 is the slow one
        t = bench.max_over_ranks(t_local)
        seqs = list(bench.rank_sequences(rank, 3))
        wl = W.WORKLOADS["tiny_mha_f32"].with_(batch=3)
        x = W.make_batch(wl, device="cpu", seqs=seqs)
        k0 = x["k"][0, 0, 0, :4].contiguous()
        got = [torch.zeros_like(k0) for _ in range(world)]
        dist.all_gather(got, k0)
        value = bench.aggregate_value(world, wl.batch, wl.n, wl.layers, t)
        out.put((rank, t, seqs, [g.tolist() for g in got], value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _run(world):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = [out.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(res)


def test_two_ranks_max_time_disjoint_sequences_and_value():
    res = _run(2)
    (r0, t0, s0, g0, v0), (r1, t1, s1, g1, v1) = res
    # every rank reports the slowest rank's time
    assert t0 == t1 == pytest.approx(2.75)
    # the ranks evict disjoint sequences that together cover the job's batch
    assert s0 == [0, 1, 2] and s1 == [3, 4, 5]
    # ... with different inputs (per-sequence seeds)
    assert g0 == g1 and g0[0] != g0[1]
    # whole-job value: both ranks' tokens over the slowest time (per layer: L = 1 here)
    assert v0 == v1 == pytest.approx(2 * 3 * 512 * 1 / (2.75 / 1e3))


def test_single_process_is_a_no_op():
    import bench
    assert bench.max_over_ranks(1.25) == 1.25
    assert list(bench.rank_sequences(0, 4)) == [0, 1, 2, 3]
