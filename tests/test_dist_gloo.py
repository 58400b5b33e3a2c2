"""The benchmark's multi-rank host logic on CPU ranks (gloo, world size 2).

Under torchrun every rank runs its own batch of tokens (weak scaling, no
data-path collective); the only cross-rank steps are the barrier around the
timed region and the max over ranks of the per-step time, from which the
whole-job throughput is computed.  These run here without a GPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        per_rank_ms = [0.8, 1.2][rank]  # rank 1 is the slow one
        dist.barrier()
        ms_max = bench.reduce_max(per_rank_ms, ws)
        value = bench.whole_job_tflops(1e12, ws, ms_max / 1e3)
        q.put((rank, ws, r, local, ms_max, value))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_whole_job_value():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ws, r, local, ms_max, value in got:
        assert ws == 2 and r == rank and local == rank
        assert ms_max == pytest.approx(1.2)  # the slowest rank sets the time
        # 2 ranks x 1 TFLOP each in 1.2 ms
        assert value == pytest.approx(2e12 / 1.2e-3 / 1e12)


def test_single_rank_is_identity():
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.whole_job_tflops(2e12, 1, 1.0) == pytest.approx(2.0)


def test_rank_batches_are_independent():
    """Each rank's tokens come from its own seed; the expert weights are shared."""
    from moe_token_dispatch_persistent_gb300 import synth

    w = synth.WORKLOADS[1]
    w1 = synth.Workload(w.name, w.T, w.H, w.F, w.E, w.k, w.seed + 1000, w.kind)
    assert not (synth.make_logits(w) == synth.make_logits(w1)).all()
    assert (synth.make_w_expert(w, 3) == synth.make_w_expert(w, 3)).all()
