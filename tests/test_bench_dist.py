"""The benchmark's multi-rank logic on CPU: two gloo ranks (no GPU).

bench.py runs one independent replica per GPU; rank 0 reports the tokens of
all ranks over the slowest rank's time. These tests run that reduction, and
the reference arm's rank-0-only output, as two local processes.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, world, port):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})


def _reduce_worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    _env(rank, world, port)
    import bench
    bench.init_dist(world, "gloo")
    # rank r takes 10*(r+1) ms for 10 steps of 1024 tokens
    job = bench.whole_job(1024, 10.0 * (rank + 1), 10, world)
    q.put((rank, job))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_whole_job_takes_the_slowest_rank_and_all_tokens():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_reduce_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        job = res[r]
        assert job["tokens"] == 2 * 1024 * 10
        assert abs(job["ms_per_step"] - 2.0) < 1e-9          # the slowest rank: 20 ms over 10 steps
        assert abs(job["value"] - 20480 / 0.020) < 1e-3


def _reference_worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    _env(rank, world, port)
    import bench
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--gpus", str(world), "--steps", "3", "--warmup", "3",
                    "--workload", "tiny"])
    q.put((rank, buf.getvalue()))


def test_reference_arm_prints_only_on_rank_zero():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_reference_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[1] == ""
    lines = [l for l in out[0].splitlines() if l.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["n_gpus"] == 2 and j["unit"] == "tokens/s"
    assert j["cpu_baseline"]["kind"] == "oracle" and j["e2e"]["h2d_bytes_per_step"] == 0
    # every key of the bench line's contract
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in j, key
    assert j["steps"] == 3 and j["warmup"] == 3 and j["higher_is_better"] is True and j["scaling"] == "weak"
    assert j["vs_baseline"] is None and j["data"] == "synthetic" and j["config"]["workload"] == "tiny"
    assert j["value"] > 0 and j["ms_per_step"] > 0
    for key in ("value", "unit", "cores", "kind", "sample"):
        assert key in j["cpu_baseline"], key
    assert j["cpu_baseline"]["value"] == j["value"] and j["cpu_baseline"]["cores"] >= 1
    assert j["e2e"]["value"] == j["value"] and j["e2e"]["unit"] == j["unit"] and j["e2e"]["d2h_bytes_per_step"] == 0
