"""The benchmark's multi-rank bookkeeping on CPU: two gloo ranks (no GPU)
reduce their timed regions to the slowest one, report the whole-job
throughput of independent replicas, and only rank 0 runs the reference arm."""
import io
import json
import os
import sys
import tempfile
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = 10.0 + 5.0 * rank                   # ms: rank 1 is the slowest
    total = bench.job_time_ms(local, world)
    value = bench.job_value(100, 8, world, total)
    # the reference arm: rank 0 alone runs and prints; the others exit without work
    buf = io.StringIO()
    if rank != 0:
        sys.argv = ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"]
        with redirect_stdout(buf):
            bench.main()
    with open(os.path.join(out_dir, "r%d.json" % rank), "w") as f:
        json.dump({"total": total, "value": value, "ref_out": buf.getvalue()}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_gloo_reduction():
    import torch.multiprocessing as mp
    world = 2
    port = 29500 + (os.getpid() % 1000)
    with tempfile.TemporaryDirectory() as d:
        ctx = mp.get_context("spawn")
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, d)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = [json.load(open(os.path.join(d, "r%d.json" % r))) for r in range(world)]
    for r in res:
        assert r["total"] == pytest.approx(15.0)                  # max over ranks
        assert r["value"] == pytest.approx(100 * 8 * 2 / 0.015)   # all ranks' tokens over the slowest time
    assert res[1]["ref_out"] == ""                                # rank 1 prints nothing for the reference arm


def test_single_rank_is_local():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_time_ms(12.5, 1) == 12.5
    assert bench.job_value(10, 8, 1, 1.0) == pytest.approx(80000.0)
