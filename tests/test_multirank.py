"""The benchmark's multi-GPU path without a GPU: two ranks over gloo on the CPU.

With N GPUs every rank runs its own replica of the workload (weak scaling; attention has no
exchange step between (b, h) slices), the ranks meet at a barrier around the timed region,
the job's time is the slowest rank's, and the throughput counts the work of all ranks. This
checks that host logic: process-group set-up from the torchrun environment, the barrier, the
max over ranks, distinct replica inputs per rank, and the whole-job throughput.
"""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      BENCH_DIST_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    from exact_attention_tcgen05_gb300 import inputs as I

    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, w)  # rank 1 is the slow one
    wl = bench.replica_workload(I.custom(1, 2, 64, 64, "bf16", True, seed=5), rank)
    q = I.make_tensor(wl, "q")
    bench.barrier(w)
    out.put((rank, slowest, wl.seed, float(q.float().sum())))
    dist.destroy_process_group()


def test_two_ranks_over_gloo():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(out.get(timeout=10) for _ in range(2))
    # every rank sees the slowest rank's time
    assert [r[1] for r in res] == [15.0, 15.0]
    # rank 0 runs the workload as seeded; rank 1 a replica with inputs of its own
    assert res[0][2] == 5 and res[1][2] != 5 and res[0][3] != res[1][3]


def test_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    # 2 TFLOP per step, 10 steps, slowest rank 4 ms in all: 5000 TFLOPS per rank's work,
    # 4 ranks -> 20000
    assert bench.job_tflops(2.0, 10, 4.0, 1) == pytest.approx(5000.0)
    assert bench.job_tflops(2.0, 10, 4.0, 4) == pytest.approx(20000.0)
