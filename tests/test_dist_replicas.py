"""The multi-process (replicas) path of bench.py on the CPU: two gloo ranks.

Decode sequences are independent problems, so N GPUs run N replicas with no
collective on the data path; the only cross-rank steps are the barrier
around the timed region and the max over ranks of the time.  This checks
those host steps with world_size 2: every rank gets the slowest rank's time,
each replica draws its own workload seed, the whole-job value counts every
replica's sequences over that time, and the reference arm's other ranks do
no work.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import synth
        slowest = bench.allreduce_max(10.0 + 5.0 * rank, world)
        bench.barrier(world)
        spec = bench.rank_spec(synth.named("decode_b8"), rank)

        class Args:
            steps, warmup, workload = 3, 1, "decode_b8"
        skipped = bench.run_reference(Args, world, rank) if rank else None
        out.put((rank, slowest, spec.seed, spec.B, spec.lengths,
                 bench.replica_value(world, spec.B, 100, slowest), skipped))
    finally:
        dist.destroy_process_group()


def test_two_gloo_replicas():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, m0, s0, b0, l0, v0, _), (r1, m1, s1, b1, l1, v1, skipped) = res
    assert m0 == m1 == 15.0                      # both ranks see the slowest time
    assert s0 != s1 and (b0, l0) == (b1, l1)     # own seed, same shapes
    assert v0 == v1 == pytest.approx(2 * 8 * 100 / 0.015)
    assert skipped is None                       # the reference arm's rank 1 returns at once
