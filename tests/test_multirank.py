"""The N > 1 path of bench.py on CPU: world-size-2 gloo groups (127.0.0.1), no GPU.

Each rank is an independent replica of the layer; the only cross-rank steps are the barrier
and the max over ranks of the timings, from which rank 0 reports the whole job's tokens/s.
The reference arm runs on rank 0 alone; the other ranks exit without work.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, timings, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        got = bench.max_over_ranks(timings[rank], dist, "cpu")
        out.put((rank, got, bench.job_tokens_per_s(world, 256, got[0])))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo():
    world, port = 2, _free_port()
    timings = [[1.25, 1.50], [1.40, 1.45]]                 # [ms, e2e_ms] per rank
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, timings, out))
             for r in range(world)]
    for p in procs:
        p.start()
    res = dict((r, (g, v)) for r, g, v in (out.get(timeout=120) for _ in range(world)))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        got, value = res[r]
        assert got == [1.40, 1.50]                          # the slowest rank decides
        assert value == pytest.approx(2 * 256 / 1.40e-3)    # all ranks' tokens / that time


def test_reference_arm_runs_on_rank_zero_only(capsys):
    from synth import layers as LY
    args = type("A", (), dict(steps=1, warmup=3, gpus=2, act="mxfp8"))()
    assert bench.run_reference(args, LY.LAYERS["tiny"], rank=1) is None
    assert capsys.readouterr().out == ""
