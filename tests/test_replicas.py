"""The N > 1 path of bench.py without GPUs: replicas as gloo ranks on CPU (world size 2).

Multi-GPU runs are replicas only -- each rank runs the whole layer on its own batch, with no data-path
collective -- so the host logic under test is what surrounds them: each rank's own batch, the max over
ranks of the step time, the whole-job throughput, and that a rank which dies ends its peers' next
reduction with an error instead of a hang.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _setup(rank, world, port):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    bench.init_replicas("gloo", timeout_s=20.0)
    return bench


def _replica_worker(rank, world, port, out_dir):
    bench = _setup(rank, world, port)
    import torch.distributed as dist
    assert bench.dist_env() == (rank, rank, world)
    ms = bench.max_over_ranks(1.0 + 2.0 * rank)  # rank 1 is the slow one
    x = bench.replica_x(0, rank, world, 4, 256)
    xs = [None] * world
    dist.all_gather_object(xs, x)
    np.save(os.path.join(out_dir, f"rank{rank}.npy"), np.array([ms, bench.job_tokens_per_s(world, 512, ms)]))
    if rank == 0:
        np.save(os.path.join(out_dir, "x.npy"), np.stack(xs))
    dist.barrier()
    dist.destroy_process_group()


def _dying_worker(rank, world, port, out_dir):
    bench = _setup(rank, world, port)
    if rank == 1:
        os._exit(3)  # a replica that dies between steps, with nothing in flight
    try:
        bench.max_over_ranks(1.0)
        outcome = "returned"
    except Exception as e:  # the peer's death surfaces as an error from the reduction
        outcome = "error: " + type(e).__name__
    with open(os.path.join(out_dir, "rank0.txt"), "w") as fh:
        fh.write(outcome)


@pytest.fixture(scope="module")
def built():
    import __graft_entry__ as g
    g.build_cpu()


def test_two_replicas_time_max_and_own_batches(built, tmp_path):
    port = _free_port()
    mp.start_processes(_replica_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    r0, r1 = np.load(tmp_path / "rank0.npy"), np.load(tmp_path / "rank1.npy")
    assert r0[0] == r1[0] == 3.0  # the slowest rank's step time
    assert r0[1] == r1[1] == 2 * 512 / 3e-3  # both replicas' tokens over that time
    xs = np.load(tmp_path / "x.npy")
    import synth
    assert np.array_equal(xs[0], synth.gen_x(0, 4, 256))  # rank 0 keeps the one-GPU batch
    assert not np.array_equal(xs[0], xs[1])  # each replica has its own tokens


def test_one_replica_alone_needs_no_process_group(built):
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5) == 2.5
    assert bench.job_tokens_per_s(1, 512, 0.5) == 512 / 0.5e-3


def test_dead_replica_ends_the_reduction_with_an_error(built, tmp_path):
    port = _free_port()
    ctx = mp.start_processes(_dying_worker, args=(2, port, str(tmp_path)), nprocs=2, join=False,
                             start_method="spawn")
    for p in ctx.processes:
        p.join(timeout=120)
    alive = [p for p in ctx.processes if p.is_alive()]
    for p in alive:
        p.kill()
    assert not alive, "a replica hung after its peer died"
    assert (tmp_path / "rank0.txt").read_text().startswith("error"), (tmp_path / "rank0.txt").read_text()
