"""bench.py's multi-rank host logic on CPU: two gloo ranks of the reference arm.

The GPU arm runs one replica per GPU and reports the slowest rank's time; its
rank handling is shared with the reference arm, which needs no GPU: rank 0
times the oracle and prints the one JSON line, every other rank exits 0 without
work.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_reference_arm_two_gloo_ranks_print_one_line():
    pytest.importorskip("torch")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--ref-seconds", "1", "--pool-blobs", "4"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = lines[0]
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 1
    assert d["value"] is not None and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_roofline_skips_a_grid_that_moves_no_bytes():
    # every read a miss: the resident gate/up grid runs with no experts and only waits
    # for SMs behind the fill, so the roofline belongs to the down grid
    sys.path.insert(0, ROOT)
    import bench
    groups = {"gemv_resident": (0, 49.0e-3 * 768, 768), "down_combine": (104_185_856 * 768, 45.4e-3 * 768, 768)}
    r = bench.roofline_from_groups(groups, 6688.8, "of measured")
    assert r["bytes_per_launch"] == 104_185_856 and r["us_per_launch"] == 45.4
    assert abs(r["frac"] - 104_185_856 / 45.4e-6 / 1e9 / 6688.8) < 1e-3
    # with no byte-moving group the largest one still gives the line
    assert bench.roofline_from_groups({"gemv_resident": (0, 1.0, 4)}, 6688.8, "of measured")["frac"] == 0.0
