"""The multi-process bench path on CPU: two gloo ranks (127.0.0.1), as torchrun would
launch them. Each rank times its own replica; rank 0 reports every rank's units over the
slowest rank's time. The reference arm under torchrun runs on rank 0 only."""
from __future__ import annotations

import io
import os
import socket
import sys
from contextlib import redirect_stdout
from pathlib import Path

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, q):
    sys.path.insert(0, str(ROOT))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_seconds = [0.5, 2.0][rank]
    slowest = bench.max_over_ranks(local_seconds, world)
    value = bench.job_throughput(1000, 10, world, slowest)
    bench.barrier(world)
    # --impl reference: only rank 0 prints; the others return without work
    buf = io.StringIO()
    args = type("A", (), dict(steps=1, warmup=0, ref_seconds=0.5))()
    with redirect_stdout(buf):
        bench.run_reference(args)
    q.put((rank, slowest, value, buf.getvalue()))
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench():
    world, port = 2, free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = {}
    for _ in range(world):
        rank, slowest, value, printed = q.get(timeout=240)
        out[rank] = (slowest, value, printed)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in range(world):
        assert out[rank][0] == 2.0                     # max over ranks
        assert out[rank][1] == pytest.approx(2 * 1000 * 10 / 2.0)
    assert '"impl": "reference"' in out[0][2]
    assert out[1][2] == ""
    # the reference arm's line carries the contract's keys: its own metric and unit, the
    # oracle as cpu_baseline (cores it used), and an e2e object with no host transfers
    import json
    line = json.loads(out[0][2].strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "config", "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["unit"] == line["unit"]


def test_oracle_split_across_threads_changes_no_bit():
    """cpu_baseline and the reference arm run the oracle on every host core by splitting
    the sample into contiguous ranges; the step is elementwise, so three steps of the split
    run must leave master, m and v identical to three steps of one call over everything."""
    sys.path.insert(0, str(ROOT))
    import numpy as np

    import bench
    n = 100_003
    one, split = bench.OracleSample(n), bench.OracleSample(n, threads=7)
    for count in (n, n - 17, n):
        one.step(count)
        split.step(count)
    for a, b in ((one.master, split.master), (one.m, split.m), (one.v, split.v)):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert one.t == split.t == 3
