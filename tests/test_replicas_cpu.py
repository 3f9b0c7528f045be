"""The multi-GPU form of the benchmark is replicas: every rank runs the layer on its own batch
(the layer has no exchange step), the job takes as long as its slowest rank, and the throughput
counts the tokens of every rank.  The rank arithmetic of bench.py is checked here with two gloo
ranks on the CPU (no GPU, no NCCL)."""
import json
import os
import socket
import subprocess
import sys

from conftest import ROOT

WORKER = r"""
import json, os, sys
sys.path.insert(0, os.environ["MOE_REPO"])
import torch.distributed as dist
import bench
rank, world = int(os.environ["RANK"]), int(os.environ["WORLD_SIZE"])
dist.init_process_group("gloo", rank=rank, world_size=world)
ms = bench.max_over_ranks(10.0 + 5.0 * rank, world)       # rank r took 10 + 5 r ms
tok_s = bench.replica_throughput(128, world, ms / 1000.0)  # 128 tokens per rank
dist.barrier()
dist.destroy_process_group()
print(json.dumps({"rank": rank, "ms": ms, "tok_s": tok_s}))
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_single_rank_is_the_value_itself():
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert bench.replica_throughput(128, 1, 0.004) == 128 / 0.004


def test_two_gloo_ranks_take_the_slowest_time_and_count_all_tokens():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), MOE_REPO=ROOT)
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    results = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        results.append(json.loads(out.strip().splitlines()[-1]))
    for r in results:
        assert r["ms"] == 15.0  # the slower rank's time, on both ranks
        assert abs(r["tok_s"] - 2 * 128 / 0.015) < 1e-6
