"""Multi-rank helpers of bench.py on CPU (gloo, world size 2).

The path runs as independent replicas, one per GPU; the only cross-rank steps
are the barrier around the timed region and the max over ranks of its time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_info()
        bench.barrier(w)
        # rank-dependent times: the max must be the slower rank's
        t = 10.0 + 5.0 * r
        results[rank] = (r, w, local, bench.max_over_ranks(t, w))
        bench.barrier(w)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_barrier_with_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        codes = [p.exitcode for p in procs]
        for p in procs:
            if p.is_alive():
                p.kill()
        assert codes == [0, 0], codes
        got = dict(results)
    assert got[0] == (0, 2, 0, 15.0)
    assert got[1] == (1, 2, 1, 15.0)


def test_single_rank_helpers_are_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)


def test_reference_arm_other_ranks_do_no_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = type("A", (), {"config": 2, "steps": 1, "warmup": 3})()
    assert bench.run_reference(args, lambda m: None) is None
