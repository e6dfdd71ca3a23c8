"""The benchmark's multi-rank path on CPU: two gloo ranks launched like the
multi-GPU run (torch.distributed.run on 127.0.0.1); the job time is the slowest
rank's, the value counts every rank's units (weak scaling), and only rank 0
prints."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_rank_aggregation_gloo():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--dist-selftest"]
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=240)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    d = json.loads(lines[0])
    assert d["n_ranks"] == 2
    assert d["max_seconds"] == 1.5           # the slower rank decides
    assert abs(d["value"] - 2 * 10.0 / 1.5) < 1e-12
    assert d["scaling"] == "weak"


def test_single_rank_aggregation():
    sys.path.insert(0, ROOT)
    import bench
    value, t = bench.aggregate(2.0, 10.0, 1)
    assert (value, t) == (5.0, 2.0)
