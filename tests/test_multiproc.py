"""Host-side multi-rank logic of bench.py, with two gloo ranks on the CPU.

The quantisation path has no exchange step: with N GPUs every rank runs the
same step on its own device (replicas).  What N > 1 adds is host logic: the
process group, the barrier around the timed region, the slowest-rank time
(max over ranks) and the whole-job rate.  These tests run that logic with two
CPU ranks, plus the reference arm's rule that only rank 0 runs and prints.
"""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("nvq_bench", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, elapsed, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    b = _bench()
    w, r, local = b.setup_dist(None, backend="gloo")
    b.barrier(w)
    slowest = b.max_over_ranks(w, elapsed[rank])
    rate = b.job_rate(w, 1_000_000_000, 4, slowest)
    b.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
        json.dump({"world": w, "rank": r, "local": local, "slowest": slowest, "rate": rate}, f)


def test_two_gloo_ranks_agree_on_slowest_time_and_job_rate(tmp_path):
    elapsed = [0.75, 1.25]
    mp.spawn(_rank_main, args=(2, _free_port(), elapsed, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(2)]
    for r, d in enumerate(res):
        assert d["world"] == 2 and d["rank"] == r and d["local"] == r
        assert d["slowest"] == 1.25                       # max over ranks, seen by both
        assert d["rate"] == pytest.approx(2 * 1e9 * 4 / 1.25 / 1e9)   # whole job, weak scaling


def test_single_rank_needs_no_process_group():
    b = _bench()
    assert b.max_over_ranks(1, 0.5) == 0.5
    b.barrier(1)
    assert b.job_rate(1, 2_000_000_000, 10, 2.0) == pytest.approx(10.0)


def _run_reference(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--steps", "1", "--warmup", "3", "--ref-frac", "1e-6"],
                          capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)


def test_reference_arm_runs_on_rank0_only():
    other = _run_reference({"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"})
    assert other.returncode == 0, other.stderr[-2000:]
    assert other.stdout.strip() == ""
    first = _run_reference({"WORLD_SIZE": "2", "RANK": "0", "LOCAL_RANK": "0"})
    assert first.returncode == 0, first.stderr[-2000:]
    line = json.loads(first.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
