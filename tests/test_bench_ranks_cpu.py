"""The benchmark's multi-rank logic (replicas, max-over-ranks timing) on CPU,
with world_size 2 over gloo.  No GPU is involved: each rank is a process."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank 0 is slow on the first timer, rank 1 on the second
        mine = [2.0 if rank == 0 else 1.0, 3.0 if rank == 1 else 0.5, float(rank)]
        got = bench.max_over_ranks(mine, dist, "cpu")
        rate = bench.whole_job_rate(world, 100.0, got[0])
        ref = bench.run_reference(None, rank, world) if rank != 0 else "skipped"
        q.put((rank, got, rate, ref))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_aggregate_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict()
    for _ in procs:
        rank, got, rate, ref = q.get(timeout=120)
        results[rank] = (got, rate, ref)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in (0, 1):
        got, rate, _ = results[rank]
        assert got == [2.0, 3.0, 1.0]          # every rank sees the slowest time
        assert rate == pytest.approx(2 * 100.0 / 2.0)  # all ranks' work over the slowest time
    assert results[1][2] is None  # non-zero ranks do no reference work and print nothing


def test_single_process_is_identity():
    assert bench.max_over_ranks([1.5, 2.5], None, "cpu") == [1.5, 2.5]
    assert bench.whole_job_rate(1, 10.0, 2.0) == 5.0


@pytest.mark.parametrize("per_copy", [262144, 64 << 20, 128 << 20, 67371008, 1 << 30, 2200000000])
def test_rotation_reads_a_copy_again_only_after_1_5_gib(per_copy):
    """Decode inputs rotate through enough cache copies that at least 1.5 GiB of
    other cache reads (12 x the 126 MB L2) separate two reads of the same copy."""
    n = bench.n_copies(per_copy)
    assert n >= 2
    assert n * per_copy >= bench.ROTATION_BYTES
    assert (n - 1) * per_copy < bench.ROTATION_BYTES or n == 2
    assert bench.ROTATION_BYTES >= 12 * 126 * 10 ** 6
