"""The multi-GPU path of the benchmark is replicas only (the pass does not
shard): each rank runs its own replica and the job's time is the slowest
rank's.  Checked here with two gloo ranks on the CPU (no GPU, no NCCL), and
the reference arm's rule that only rank 0 runs and prints."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_RANK = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import torch.distributed as dist
dist.init_process_group("gloo")
import bench
rank, world = dist.get_rank(), dist.get_world_size()
t = bench.job_seconds(1.0 + 0.5 * rank, world, "cpu")
print(json.dumps({"rank": rank, "t": t, "value": bench.job_value(2e9, 10, world, t)}))
dist.destroy_process_group()
"""


def _port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_replicas_report_the_slowest_rank():
    port = _port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), LOCAL_RANK=str(r))
        procs.append(subprocess.Popen([sys.executable, "-c", _RANK, ROOT], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=180)
        assert p.returncode == 0, err[-2000:]
        outs.append(json.loads(out.strip().splitlines()[-1]))
    for o in outs:
        assert o["t"] == 1.5                      # the slower rank's time, on both ranks
        assert abs(o["value"] - 2e9 * 10 * 2 / 1.5 / 1e9) < 1e-9


def test_single_process_time_is_its_own():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_seconds(2.5, 1, "cpu") == 2.5
    assert bench.job_value(1e9, 4, 1, 2.0) == 2.0


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
