"""bench.py's multi-process path on CPU: two ranks over gloo (no GPU).

The decode path shards by sequence with no data-path collective; with N
processes each rank runs its own replica and bench.py only combines the
timings: the whole-job rate is the units of all ranks over the slowest
rank's time, and every rank gets the same answer. Under torchrun the
reference arm runs on rank 0 alone; the other ranks leave without work or
output.
"""
import contextlib
import io
import os
import socket
import types

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    try:
        w, r, local = bench.dist_env()
        dist = bench.init_dist(w, "gloo")
        bench.barrier(dist)
        # rank r processed 16 * (r + 1) tokens in 10 + r ms
        rate, ms = bench.whole_job_rate(16 * (r + 1), 10.0 + r, dist)
        mx = bench.max_over_ranks(float(r), dist)
        sm = bench.sum_over_ranks(1.0, dist)
        bench.barrier(dist)
        dist.destroy_process_group()
        q.put((r, w, local, rate, ms, mx, sm))
    except Exception as e:  # reported to the parent, which fails the test
        q.put((rank, "error", repr(e)))


@pytest.mark.timeout(120)
def test_two_gloo_ranks_agree_on_the_whole_job_rate():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=100) for _ in range(world)]
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    for res in results:
        assert res[1] != "error", res
    want_ms = 11.0
    want_rate = (16 + 32) / (want_ms / 1e3)
    for r, w, local, rate, ms, mx, sm in results:
        assert w == world and local == r
        assert ms == want_ms and abs(rate - want_rate) < 1e-9 * want_rate
        assert mx == 1.0 and sm == 2.0


def test_single_process_helpers_are_identities():
    assert bench.init_dist(1, "gloo") is None
    assert bench.whole_job_rate(32, 4.0, None) == (32 / 0.004, 4.0)
    assert bench.max_over_ranks(3.5, None) == 3.5 and bench.sum_over_ranks(2, None) == 2.0


def test_reference_arm_runs_on_rank_zero_only():
    args = types.SimpleNamespace(workload="dsv2_b16_l4096", steps=3, warmup=1)
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        assert bench.run_reference(args, 2, 1) is None
    assert out.getvalue() == ""


@pytest.mark.timeout(240)
def test_gpus_flag_starts_one_process_per_rank():
    """``bench.py --gpus 2`` outside torchrun starts two local ranks itself
    (torch.distributed.run on 127.0.0.1); the reference arm, which needs no
    GPU, then prints exactly one line, from rank 0, for the whole job."""
    import json
    import subprocess
    import sys
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, bench.__file__, "--gpus", "2", "--impl", "reference",
                        "--workload", "tiny_fp32", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=220, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2
