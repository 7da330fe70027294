"""Multi-rank host logic of bench.py, world size 2 over gloo on the CPU (no GPU).

The path has no exchange step: under torchrun every rank runs its own replica
of the workload and rank 0 reports the slowest rank's time (max over ranks)
and the whole job's throughput.  These tests run that logic with two real
processes and a gloo process group on 127.0.0.1.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, os, sys
sys.path.insert(0, {root!r})
import torch
torch.cuda.is_available = lambda: False      # force the gloo backend
import bench
ws, rank, local = bench.dist_env()
dist = bench.make_group(ws)
t = bench.max_over_ranks(dist, 1.5 * (rank + 1))
bench.barrier(dist)
v = bench.job_throughput(1000, ws, t)
print(json.dumps({{"rank": rank, "ws": ws, "local": local, "max": t, "value": v}}))
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _run_ranks(script, ws=2, extra_env=None, timeout=120):
    port = _free_port()
    procs = []
    for r in range(ws):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(r),
                   WORLD_SIZE=str(ws), LOCAL_RANK=str(r), CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        procs.append(subprocess.Popen([sys.executable, "-c", script], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            o, e = p.communicate(timeout=timeout)
        except subprocess.TimeoutExpired:
            p.kill()
            raise
        assert p.returncode == 0, e[-2000:]
        outs.append(o)
    return outs


def test_max_over_ranks_and_job_throughput_gloo():
    outs = _run_ranks(WORKER.format(root=ROOT))
    recs = sorted((json.loads(o.strip().splitlines()[-1]) for o in outs), key=lambda d: d["rank"])
    assert [d["rank"] for d in recs] == [0, 1]
    for d in recs:
        assert d["ws"] == 2 and d["local"] == d["rank"]
        assert d["max"] == pytest.approx(3.0)            # the slower rank's time, on every rank
        # whole-job throughput: units of all ranks over the slowest rank's time (ms)
        assert d["value"] == pytest.approx(2 * 1000 / 3.0e-3)


def test_reference_arm_runs_on_rank_zero_only():
    script = (f"import sys; sys.path.insert(0, {ROOT!r}); import bench, argparse; "
              "bench.bench_reference(argparse.Namespace(steps=1, warmup=0, gpus=2))")
    out = subprocess.run([sys.executable, "-c", script], cwd=ROOT, capture_output=True, text=True, timeout=120,
                         env=dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1"))
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip() == ""                      # rank 1: no work, no line
