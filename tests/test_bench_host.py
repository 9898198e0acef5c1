"""Host-side logic of bench.py that needs no GPU: the max-over-ranks timing
reduction and whole-job throughput of the N > 1 (replica) path, run as two
gloo ranks on the CPU, and the reference (CPU oracle) arm's launch contract."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

RANK_SCRIPT = r"""
import json, os, sys
sys.path.insert(0, {root!r})
import torch.distributed as td
import bench
td.init_process_group("gloo")
r = td.get_rank()
ms = 10.0 + 5.0 * r                      # rank 1 is the slow one
got = bench.max_over_ranks(ms)
gbs = bench.whole_job_gbs(td.get_world_size(), 4, 1_000_000_000, got)
td.barrier()
td.destroy_process_group()
print(json.dumps({{"rank": r, "max_ms": got, "gbs": gbs}}))
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_without_group_is_identity():
    assert bench.max_over_ranks(3.25) == 3.25


def test_whole_job_gbs_counts_every_rank():
    # 2 ranks x 3 steps x 2 GB in 1.5 s of the slowest rank = 8 GB/s
    assert bench.whole_job_gbs(2, 3, 2_000_000_000, 1500.0) == pytest.approx(8.0)


def test_two_gloo_ranks_take_the_slowest_time():
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE="2", LOCAL_RANK=str(r),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_SCRIPT.format(root=ROOT)],
                                      env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["max_ms"] == 15.0
        # 2 ranks x 4 steps x 1 GB / 15 ms
        assert o["gbs"] == pytest.approx(2 * 4 / 0.015)


def _run_bench(args, **env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], env=env,
                          capture_output=True, text=True, timeout=300)


def test_reference_arm_other_ranks_exit_without_work():
    r = _run_bench(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"],
                   RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_prints_contract_line():
    r = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "3",
                    "--ref-step-seconds", "0.5"])
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["config"]["workload"]


def test_warmup_below_three_is_refused():
    r = _run_bench(["--steps", "1", "--warmup", "2"])
    assert r.returncode != 0
    assert "warmup" in r.stderr
