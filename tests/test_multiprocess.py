"""Multi-process path of bench.py on CPU: two ranks over gloo (world size 2).

The bench runs one replica of the workload per rank (the B x H sequences are independent, so
the path has no data-path collective); the only collectives are the timing barrier and the
max-over-ranks reduction, and the reported value is the whole job's units over the slowest
rank's time.  These tests run exactly those helpers in two processes, and check that the
reference arm does its work on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


_RANK_SCRIPT = r"""
import json, os, sys
sys.path.insert(0, {root!r})
import bench
world, rank, local = bench.dist_setup()
bench.barrier(world)
# rank r took (r + 1) ms for 1000 units: the job rate is 2000 units / 2 ms
value, ms = bench.aggregate_rate(1000.0, float(rank + 1), world)
mx = bench.max_over_ranks(10.0 * rank - 3.0, world)
bench.barrier(world)
import torch.distributed as dist
backend = dist.get_backend()
dist.destroy_process_group()
print(json.dumps({{"rank": rank, "world": world, "value": value, "ms": ms, "max": mx,
                  "backend": backend}}))
"""


def _launch(script: str, world: int, extra_env=None, args=()):
    port = _free_port()
    procs = []
    for r in range(world):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(world),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", script, *args], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True, cwd=ROOT))
    outs = []
    for p in procs:
        try:
            out, err = p.communicate(timeout=240)
        except subprocess.TimeoutExpired:
            p.kill()
            raise
        assert p.returncode == 0, err[-2000:]
        outs.append(out)
    return outs


def test_two_rank_timing_helpers_over_gloo():
    outs = _launch(_RANK_SCRIPT.format(root=ROOT), 2)
    res = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    for r in res:
        assert r["world"] == 2 and r["backend"] == "gloo"
        assert r["ms"] == pytest.approx(2.0)          # slowest rank
        assert r["value"] == pytest.approx(1.0e6)     # 2 x 1000 units / 2 ms
        assert r["max"] == pytest.approx(7.0)         # max(-3, 7)
    assert sorted(r["rank"] for r in res) == [0, 1]


_REF_SCRIPT = r"""
import os, sys, runpy
sys.path.insert(0, {root!r})
sys.argv = ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"]
runpy.run_path(os.path.join({root!r}, "bench.py"), run_name="__main__")
"""


def test_reference_arm_runs_on_rank_zero_only():
    outs = _launch(_REF_SCRIPT.format(root=ROOT), 2)
    lines = [[l for l in o.strip().splitlines() if l.startswith("{")] for o in outs]
    assert len(lines[0]) == 1 and lines[1] == []
    line = json.loads(lines[0][0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    # the line keeps the contract's keys: the same metric and unit as the kernel arm, the
    # oracle described as its CPU baseline, and an end-to-end figure with no device copies
    for key in ("metric", "unit", "higher_is_better", "ms_per_step", "config", "dtype", "data"):
        assert key in line, key
    assert line["higher_is_better"] is True and line["unit"] == "tokens/s"
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == line["value"]
    assert cpu["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
