"""Host-side logic of the N > 1 benchmark path, run as two gloo ranks on CPU:
the job time is the slowest rank's, the throughput counts every replica, and
only rank 0 prints the reference arm's line."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, os, sys
sys.path.insert(0, os.environ["ROOT"])
import torch.distributed as dist
import bench
rank = int(os.environ["RANK"]); world = int(os.environ["WORLD_SIZE"])
dist.init_process_group("gloo")
ms = 100.0 + 50.0 * rank                      # rank 1 is the slower replica
mx = bench.reduce_max_ms(ms, world)
val = bench.whole_job_tflops(world, 1e12, 10, mx)
dist.barrier()
print(json.dumps({"rank": rank, "max": mx, "value": val}))
dist.destroy_process_group()
"""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(code, world=2, extra_env=None, args=()):
    port = _free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, ROOT=ROOT, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        env.update(extra_env or {})
        cmd = [sys.executable, "-c", code] if code else [sys.executable, os.path.join(ROOT, "bench.py"), *args]
        procs.append(subprocess.Popen(cmd, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=240)
        assert p.returncode == 0, err
        outs.append(out)
    return outs


def test_max_over_ranks_and_whole_job_throughput():
    outs = _launch(WORKER)
    res = [json.loads(o.strip().splitlines()[-1]) for o in outs]
    for r in res:
        assert r["max"] == 150.0                                  # the slowest rank
        assert r["value"] == pytest.approx(2 * 1e12 * 10 / 0.150 / 1e12)


def test_reference_arm_prints_on_rank0_only():
    outs = _launch(None, args=("--impl", "reference", "--steps", "1", "--warmup", "0", "--gpus", "2"))
    lines0 = [l for l in outs[0].splitlines() if l.startswith("{")]
    lines1 = [l for l in outs[1].splitlines() if l.startswith("{")]
    assert len(lines0) == 1 and not lines1
    line = json.loads(lines0[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
