"""The benchmark's multi-rank logic on CPU with the gloo backend (two ranks):
the slowest rank's time decides, whole-job throughput counts every rank's
batch, and only rank 0 reports.  The data path itself has no collective
(each rank convolves its own batch)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as tdist
    import bench
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        worst = bench.reduce_max(local_ms)
        bench.barrier()
        tops = bench.weak_scaling_tops(world, steps=4, ops_per_step=1e12, max_ms=worst)
        out[rank] = (worst, tops)
    finally:
        tdist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    # 2 ranks x 4 steps x 1e12 ops in 15 ms
    assert res[0][1] == pytest.approx(2 * 4 * 1e12 / 15e-3 / 1e12)


def _ref_worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import bench
    import io
    import contextlib
    args = type("A", (), {"workload": "small_i8_16x16x32", "steps": 1, "warmup": 0})()
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, rank, world)
    out[rank] = buf.getvalue()


def test_reference_arm_reports_on_rank_zero_only():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_ref_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[1] == ""
    import json
    line = json.loads(res[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 2
