"""The bench's multi-process path on the CPU: two ranks over gloo.

The hot path has no exchange step, so N GPUs run N independent replicas;
what crosses ranks is the timing (max over ranks), the work (sum over
ranks) and, for the reference arm, the rule that rank 0 alone works and
prints.  Each test starts real processes with the launcher's environment
(MASTER_ADDR 127.0.0.1, RANK, WORLD_SIZE, LOCAL_RANK)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


RANK_SCRIPT = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import bench
rank, local, ws = bench.dist_setup(None)
t = [2.0, 3.0][rank]                      # this rank's ms per step
rate, ms_max = bench.aggregate(1e12, 5, t, ws)
out = {"rank": rank, "ws": ws, "local": local, "max": bench.reduce_max(10.0 * (rank + 1), ws),
       "sum": bench.reduce_sum(rank + 1.0, ws), "rate": rate, "ms_max": ms_max}
bench.barrier(ws)
import torch.distributed as dist
dist.destroy_process_group()
print(json.dumps(out))
"""


def test_two_rank_reductions_and_aggregate():
    port = free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(r), WORLD_SIZE="2",
                   LOCAL_RANK=str(r))
        procs.append(subprocess.Popen([sys.executable, "-c", RANK_SCRIPT, ROOT], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        so, se = p.communicate(timeout=180)
        assert p.returncode == 0, se[-2000:]
        outs.append(json.loads(so.strip().splitlines()[-1]))
    for o in outs:
        assert o["ws"] == 2
        assert o["max"] == 20.0
        assert o["sum"] == 3.0
        # 2 ranks x 5 steps x 1e12 units over the slower rank's 5 x 3 ms
        assert o["ms_max"] == 3.0
        assert o["rate"] == pytest.approx(2 * 5 * 1e12 / (5 * 3e-3), rel=1e-12)
    assert sorted(o["rank"] for o in outs) == [0, 1]


def test_single_rank_aggregate_is_local():
    sys.path.insert(0, ROOT)
    import bench
    rate, ms_max = bench.aggregate(4.0, 10, 2.0, 1)
    assert ms_max == 2.0 and rate == pytest.approx(4.0 * 10 / (10 * 2e-3))


def test_reference_arm_under_torchrun_two_ranks():
    """The driver's launch of the reference arm at N = 2: exactly one JSON
    line, from rank 0, and both ranks exit 0."""
    from oracle.build import build_oracle
    build_oracle()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(free_port()), os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-3000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0
