"""The multi-GPU path of bench.py is replicas only (no data-path collective): one process per GPU,
a barrier around the timed region, the job's time is the slowest rank's, and the value is the units
all ranks processed over that time.  Here the host side of that logic runs as two gloo ranks on the
CPU: max over ranks, the whole-job rate, and the reference arm doing its work on rank 0 alone."""
import contextlib
import io
import multiprocessing as mp
import os
import socket
import sys

import pytest

from conftest import ROOT

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, loc = bench.rank_info()
    ms = bench.max_over_ranks(dist, 1.0 + 2.0 * rank, "cpu")        # rank 0 took 1 ms, rank 1 took 3 ms
    rate = bench.job_rate(w, 1000, ms)
    printed = ""
    if rank == 1:   # the reference arm runs on rank 0 only: rank 1 returns at once and prints nothing
        args = bench.parse_args(["--impl", "reference", "--steps", "3", "--warmup", "3"])
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            bench.run_reference(args)
        printed = buf.getvalue()
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, r, w, loc, ms, rate, printed))


def test_two_gloo_replicas_agree_on_time_and_rate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_replica, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, r_env, w, loc, ms, rate, printed) in enumerate(results):
        assert (r, r_env, w, loc) == (rank, rank, world, rank)
        assert ms == 3.0                                   # the slowest rank sets the job's time
        assert rate == pytest.approx(2 * 1000 / 3e-3)      # all ranks' units over that time
        assert printed == ""


def test_single_process_needs_no_collective():
    import bench
    assert bench.max_over_ranks(None, 2.5) == 2.5
    assert bench.job_rate(1, 16384, 0.5) == pytest.approx(16384 / 0.5e-3)
