"""The N > 1 benchmark path on the CPU: two gloo ranks.

bench.py runs one independent replica per GPU (the layer shards into
independent column blocks, so there is no data-path exchange); ranks meet only
at barriers, and rank 0 reports the slowest rank's time. These tests run that
host logic with world_size 2 over gloo, without a GPU.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch
    import torch.distributed as dist
    import bench
    w, r, _ = bench.setup_dist()
    assert (w, r) == (world, rank)
    # slowest rank wins
    t = bench.max_over_ranks(0.5 + rank, world, torch.device("cpu"))
    bench.barrier(world)
    # the reference arm prints on rank 0 only
    buf = io.StringIO()
    args = type("A", (), {"steps": 1, "warmup": 0})()
    with redirect_stdout(buf):
        if rank != 0:
            bench.reference(args)
    q.put((rank, t, buf.getvalue()))
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_rank_max_and_rank0_only_output():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [1.5, 1.5]
    assert out[1][2] == ""  # rank 1 printed nothing


def test_reference_arm_line_format():
    sys.path.insert(0, ROOT)
    import bench
    buf = io.StringIO()
    args = type("A", (), {"steps": 1, "warmup": 0})()
    os.environ.pop("RANK", None)
    os.environ.pop("WORLD_SIZE", None)
    with redirect_stdout(buf):
        bench.reference(args)
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
