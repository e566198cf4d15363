"""bench.py on the CPU: the reference arm of every workload prints one JSON line
of the contract, and the multi-process plumbing (torchrun, gloo, world size 2)
prints one line from rank 0 with the other rank exiting cleanly; the
max-over-ranks timing helper agrees across ranks."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
        "cpu_baseline", "e2e")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _json_lines(out):
    return [json.loads(l) for l in out.splitlines() if l.strip().startswith("{")]


def _env():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", MASTER_ADDR="127.0.0.1",
               OMP_NUM_THREADS="1")
    env.pop("WORLD_SIZE", None)
    env.pop("RANK", None)
    return env


@pytest.mark.parametrize("workload", ["layer", "sampler", "rmsnorm", "linear"])
def test_reference_arm_prints_the_contract_line(workload):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", workload, "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, env=_env(), cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    line = lines[0]
    for k in KEYS:
        assert k in line, k
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["unit"] == line["unit"]
    assert "workload" in line["config"]


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "2", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=_env(), cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2 and lines[0]["impl"] == "reference"


_RANKS = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
world, rank, local = bench.dist_setup(2)
assert dist.get_backend() == "gloo"
bench.barrier(world)
v = bench.max_over_ranks(world, 1.5 + rank)
bench.barrier(world)
with open(os.path.join({out!r}, "rank%d.json" % rank), "w") as f:
    json.dump({{"rank": rank, "max": v}}, f)
dist.destroy_process_group()
"""


def test_max_over_ranks_with_gloo(tmp_path):
    port = _free_port()
    script = tmp_path / "ranks.py"
    script.write_text(_RANKS.format(root=ROOT, out=str(tmp_path)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), str(script)]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=_env(), cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    got = {}
    for k in (0, 1):
        d = json.loads((tmp_path / f"rank{k}.json").read_text())
        got[d["rank"]] = d["max"]
    assert got == {0: 2.5, 1: 2.5}
