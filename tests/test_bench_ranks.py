"""bench.py's multi-rank logic on CPU: world size 2 over gloo.

The timed region's duration is the maximum over ranks and the job's
throughput the sum of the units every rank processed; each replica rank
draws its own batch; under the reference arm only rank 0 runs and prints.
"""

import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    bench.init_dist(world, "gloo")
    try:
        mx = bench.max_over_ranks(10.0 + 5 * rank, world)
        sm = bench.sum_over_ranks(100.0 * (rank + 1), world)
        seeds = bench.rank_seed(4, rank)
        bench.barrier(world)
        buf = io.StringIO()
        with redirect_stdout(buf):
            bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1",
                                                  "--warmup", "0", "--cpu-sample", "4096",
                                                  "--n", "1024"]))
        q.put((rank, mx, sm, seeds, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_over_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = {}
    for _ in range(world):
        rank, mx, sm, seed, out = q.get(timeout=240)
        results[rank] = (mx, sm, seed, out)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results[0][0] == results[1][0] == 15.0          # slowest rank sets the time
    assert results[0][1] == results[1][1] == 300.0         # units of every rank count
    assert results[0][2] != results[1][2]                  # replicas draw their own batch
    assert '"impl": "reference"' in results[0][3]          # rank 0 prints the reference line
    assert results[1][3] == ""                             # the other rank prints nothing


def test_reference_line_fields():
    """The reference arm's JSON line at one rank: the step's metric and unit,
    the oracle as its CPU baseline, and an end-to-end figure equal to its
    value with no host-device copies."""
    import json
    sys.path.insert(0, ROOT)
    import bench
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "2", "--warmup", "1",
                                              "--cpu-sample", "16384", "--n", "8192"]))
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "Gelem/s"
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["n_gpus"] == 1 and line["steps"] == 2 and line["warmup"] == 1
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == line["value"]
    assert "4096 elements" in cb["sample"]  # min(cpu_sample / 4, n)
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert line["config"]["sample_n"] == 4096 and line["config"]["n"] == 8192
