"""Host-side logic of the multi-GPU benchmark path, on CPU with gloo (world size 2):
each rank owns a full batch (weak scaling, no data-path collective); the job's
time is the max over ranks."""
import os
import socket

import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    r, w, local = bench.dist_env()
    d = bench.dist_init(w, "gloo")
    times = {0: 12.5, 1: 17.25}
    worst = bench.max_over_ranks(times[r], d)
    bench.barrier(d)
    q.put((r, w, local, worst))
    d.destroy_process_group()


def test_two_rank_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 2 and g[3] == 17.25 for g in got)
    assert [g[2] for g in got] == [0, 1]


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.0, None) == 3.0
    bench.barrier(None)


def _e2e_worker(rank, world, port, q):
    import torch
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), LOCAL_WORLD_SIZE=str(world))
    d = bench.dist_init(world, "gloo")
    if rank == 1:  # this rank's host has no room for its pinned buffers
        bench.host_available_bytes = lambda: 1
    x = {n: torch.zeros(8) for n in ("q", "k", "v", "g", "beta")}
    res = bench.run_e2e(None, None, x, 1, torch.zeros(8), torch.zeros(1), None, None, d, world)
    bench.barrier(d)  # no rank is left waiting inside the leg
    q.put((rank, res.get("value"), res.get("unavailable", "")))
    d.destroy_process_group()


def test_e2e_leg_is_left_by_all_ranks_together():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_e2e_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] is None and g[2].startswith("host memory") for g in got)
