"""The benchmark's multi-process host logic on CPU: two ranks over the gloo backend (one
process per GPU on a GPU machine; replicas only, so the ranks exchange nothing but timings)."""
import json
import os
import socket
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r"""
import json, os, sys, time
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
world, rank, local = bench._dist_env()
dist.init_process_group("gloo")
# each replica "times" a step of its own; the job reports the slowest one
mine = [1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)]
dist.barrier()
agg = bench.max_over_ranks(mine, world)
dist.barrier()
print(json.dumps({{"rank": rank, "world": world, "local": local, "agg": agg,
                  "value": bench.job_tokens_per_s(8192, world, agg[0])}}), flush=True)
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_agree_on_the_slowest_replica():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_SCRIPT.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    assert sorted(o["rank"] for o in outs) == [0, 1]
    for o in outs:
        assert o["world"] == 2 and o["local"] == o["rank"]
        assert o["agg"] == [2.0, 5.0, 0.5]            # element-wise maximum over the ranks
        assert abs(o["value"] - 8192 * 2 / 2e-3) < 1e-6  # all tokens / slowest step (2 ms)


def test_single_process_needs_no_process_group():
    assert bench.max_over_ranks([3, 1.5], 1) == [3.0, 1.5]
    assert bench.job_tokens_per_s(8192, 1, 0.5) == 8192 / 0.5e-3


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    """Under torchrun only rank 0 times the oracle and prints; the other ranks exit 0 at once."""
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"]) == 0
    assert capsys.readouterr().out == ""
