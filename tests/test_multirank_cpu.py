"""The benchmark's multi-rank logic on the CPU: two gloo ranks.

On GPUs every rank runs its own replica of the workload (the simulated
group does not span GPUs); the only cross-rank steps are the barrier, the
maximum of the timed region over ranks, and printing on rank 0 alone."""
import contextlib
import io
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), OMP_NUM_THREADS="1")
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from synth.workloads import CFG1
    slowest = bench.max_over_ranks(10.0 + rank)
    dist.barrier()
    buf = io.StringIO()

    class Args:
        gpus, steps, warmup = world, 1, 0

    with contextlib.redirect_stdout(buf):
        bench.run_reference(Args, CFG1.replace(numels=(4096,)))
    out.put((rank, slowest, buf.getvalue()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_rank0_output():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        rank, slowest, text = q.get(timeout=300)
        res[rank] = (slowest, text)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][0] == res[1][0] == 11.0
    assert '"impl": "reference"' in res[0][1]
    assert res[1][1] == ""


def test_single_process_max_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
