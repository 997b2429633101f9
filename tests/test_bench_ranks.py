"""The benchmark's multi-rank host logic on CPU: two gloo ranks launched like torchrun
(RANK / WORLD_SIZE / LOCAL_RANK / MASTER_* in the environment) agree on the slowest rank's
time, and the whole-job value counts every rank's bytes once over that time."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import os, sys, json
sys.path.insert(0, os.environ["KV_ROOT"])
import torch, torch.distributed as dist
import bench
rank, world, local = bench.dist_env()
dist.init_process_group("gloo")
ms = bench.max_over_ranks(torch, 1.0 + 2.0 * rank, world, "cpu")
value = bench.whole_job_gbs(1_000_000, world, ms)
dist.barrier()
print(json.dumps({"rank": rank, "world": world, "local": local, "ms": ms, "value": value}), flush=True)
dist.destroy_process_group()
"""


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_take_the_slowest_time():
    pytest.importorskip("torch.distributed")
    port = free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE="2", LOCAL_RANK=str(r), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), KV_ROOT=ROOT)
        procs.append(subprocess.Popen([sys.executable, "-c", CHILD], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(out.strip().splitlines()[-1])
    import json
    got = sorted((json.loads(o) for o in outs), key=lambda d: d["rank"])
    assert [d["local"] for d in got] == [0, 1] and all(d["world"] == 2 for d in got)
    # rank 1 took 3 ms: both ranks report it, and the value is 2 x 1 MB / 3 ms
    assert all(d["ms"] == 3.0 for d in got)
    assert all(abs(d["value"] - 2e6 / 3e-3 / 1e9) < 1e-12 for d in got)


def test_single_rank_defaults():
    import bench
    saved = {k: os.environ.pop(k, None) for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    try:
        assert bench.dist_env() == (0, 1, 0)
        import torch
        assert bench.max_over_ranks(torch, 2.5, 1, "cpu") == 2.5
        assert bench.whole_job_gbs(67108864, 1, 0.01) == pytest.approx(6710.8864)
    finally:
        for k, v in saved.items():
            if v is not None:
                os.environ[k] = v
