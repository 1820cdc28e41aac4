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
    with mp.get_context("spawn").Manager() as mgr:
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
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_ref_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[1] == ""
    import json
    line = json.loads(res[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 2


# ---------------------------------------------------------------- batch shards
def test_shard_range_covers_the_batch():
    import bench
    for n in (1, 2, 5, 7, 32, 256):
        for world in range(1, min(n, 9) + 1):
            ranges = [bench.shard_range(n, world, r) for r in range(world)]
            assert ranges[0][0] == 0 and ranges[-1][1] == n
            for (lo, hi), (lo2, _) in zip(ranges, ranges[1:]):
                assert hi == lo2                      # consecutive and disjoint
            sizes = [hi - lo for lo, hi in ranges]
            assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        bench.shard_range(3, 4, 0)                    # fewer images than ranks
    with pytest.raises(ValueError):
        bench.shard_range(8, 2, 2)                    # no such rank


SHARD_CASE = dict(seed=9100, N=5, H=9, W=7, C=16, K=32, R=3, S=3)


def _shard_worker(rank, world, port, out):
    """Each rank convolves its images of one batch with the oracle; rank 0
    gathers the shards in rank order."""
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as tdist
    import bench
    import fconv_inputs as FI
    import oracle
    c = SHARD_CASE
    P, _, _ = oracle.out_geometry(c["H"], c["R"], 1, oracle.SAME)
    Q, _, _ = oracle.out_geometry(c["W"], c["S"], 1, oracle.SAME)
    inp = FI.random_case(c["seed"], c["N"], c["H"], c["W"], c["C"], c["K"], c["R"], c["S"],
                         "int8", (P, Q), True)
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        lo, hi = bench.shard_range(c["N"], world, rank)
        y, _ = oracle.fused_conv_i8(inp["x"][lo:hi], inp["w"], inp["bias"], inp["side"][lo:hi],
                                    0.002, 0.5, True, 1, oracle.SAME)
        shards = [None] * world
        tdist.all_gather_object(shards, (lo, hi, y))
        if rank == 0:
            out["shards"] = shards
            out["full"] = oracle.fused_conv_i8(inp["x"], inp["w"], inp["bias"], inp["side"],
                                               0.002, 0.5, True, 1, oracle.SAME)[0]
    finally:
        tdist.destroy_process_group()


def test_batch_shards_reassemble_the_unsharded_result():
    import numpy as np
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_shard_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    shards = res["shards"]
    assert [(lo, hi) for lo, hi, _ in shards] == [(0, 2), (2, 5)]
    whole = np.concatenate([y for _, _, y in shards], axis=0)
    assert np.array_equal(whole, res["full"])
