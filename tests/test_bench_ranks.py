"""The benchmark's multi-rank arithmetic on CPU with the gloo backend
(world size 2): the job time is the slowest rank's, the value counts every
rank's units, and the reference arm prints only on rank 0."""
import json
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [12.5, 20.0][rank]
        t = bench.max_over_ranks(ms, dist, torch.device("cpu"))
        v = bench.job_value(1000, 10, t, world)
        dist.barrier()
        out[rank] = (t, v)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn")
        res = dict(out)
    assert res[0] == res[1] == (20.0, 2 * 1000 * 10 / 20e-3)


def test_reference_arm_prints_on_rank_zero_only(capsys):
    import synth

    class Args:
        steps, warmup, gpus = 1, 0, 2

    shape = synth.SHAPES["tiny"]
    bench.run_reference(Args, shape, rank=1, world=2)
    assert capsys.readouterr().out == ""
    bench.run_reference(Args, shape, rank=0, world=2)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
