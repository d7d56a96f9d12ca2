"""The bench's multi-rank host logic on two CPU processes over gloo.

A run on N GPUs is N replicas of the step (no data-path collective): the
ranks meet only at the barriers around each timed region and in the max
over ranks of its duration; rank 0 alone prints the JSON line, and the
reference arm (the oracle on the host cores) runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

# one rank: a timed region bracketed by barriers, each rank taking a
# different time, then the max over ranks and the rank-0 line
CHILD = r"""
import io, json, sys, time
sys.path.insert(0, sys.argv[1])
import bench
r = bench.Ranks("gloo")
r.barrier()
t0 = time.perf_counter()
time.sleep(0.05 + 0.25 * r.rank)          # rank 1 is the slow one
ms = (time.perf_counter() - t0) * 1e3
r.barrier()
mx = r.max(ms)
r.emit({"rank": r.rank, "own_ms": ms, "max_ms": mx,
        "value": bench.job_tflops(r.world, 1e12, mx)})
sys.stderr.write(json.dumps({"rank": r.rank, "own_ms": ms, "max_ms": mx}) + "\n")
r.close()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, world, port):
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
               WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    env.pop("CUDA_VISIBLE_DEVICES", None)
    return env


def test_two_ranks_max_over_ranks_and_one_line():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", CHILD, ROOT], env=_env(r, 2, port),
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True) for r in range(2)]
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=120)
        finally:
            if p.poll() is None:
                p.kill()
        assert p.returncode == 0, err
        outs.append((out, err))
    seen = [json.loads(e.strip().splitlines()[-1]) for _, e in outs]
    slow = max(s["own_ms"] for s in seen)
    # both ranks agree on the max, and it is the slow rank's own time
    assert all(s["max_ms"] == slow for s in seen)
    assert slow >= 300.0 - 1.0
    # rank 0 prints exactly one line, rank 1 nothing
    lines0 = outs[0][0].strip().splitlines()
    assert len(lines0) == 1 and outs[1][0] == ""
    line = json.loads(lines0[0])
    assert line["max_ms"] == slow
    # whole-job value: both replicas' work over the slowest rank's time
    assert line["value"] == pytest.approx(2 * 1e12 / (slow / 1e3) / 1e12)


def test_job_tflops_closed_form():
    # 4 replicas of 2 TFLOP each in 0.5 ms: 8 TFLOP / 0.5 ms = 16 PFLOP/s
    assert bench.job_tflops(4, 2e12, 0.5) == pytest.approx(16000.0)
    assert bench.job_tflops(1, 1e9, 1.0) == pytest.approx(1.0)


def test_single_rank_needs_no_process_group(monkeypatch, capsys):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    r = bench.Ranks("gloo")
    assert (r.world, r.rank, r.dist) == (1, 0, None)
    r.barrier()
    assert r.max(3.5) == 3.5
    r.emit({"a": 1})
    assert json.loads(capsys.readouterr().out) == {"a": 1}
    r.close()


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the reference arm's other ranks exit 0 at once, print
    nothing and do no work."""
    t0 = time.perf_counter()
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], env=_env(1, 2, _free_port()), capture_output=True, text=True, timeout=120)
    assert p.returncode == 0, p.stderr
    assert p.stdout == ""
    assert time.perf_counter() - t0 < 60.0
