"""bench.py's multi-rank host logic on CPU: world_size 2 over gloo (no GPU).

With N > 1 every rank runs its own replica of the workload; the timed region
is bracketed by barriers, the time is the max over ranks and the value is the
sum of the ranks' work over that time.  These tests run the same helpers as
bench.py under two spawned gloo ranks.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import time
    import bench
    dist = bench.init_dist(world, "gloo")
    bench.barrier(dist, device_sync=False)
    t0 = time.perf_counter()
    time.sleep(0.05 * (rank + 1))          # rank 1 is the slow one
    elapsed = time.perf_counter() - t0
    bench.barrier(dist, device_sync=False)
    worst = bench.max_over_ranks(dist, elapsed)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"elapsed": elapsed, "worst": worst}, f)
    dist.destroy_process_group()


def test_max_over_ranks_gloo(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    r0 = json.load(open(tmp_path / "r0.json"))
    r1 = json.load(open(tmp_path / "r1.json"))
    assert r0["worst"] == r1["worst"] == pytest.approx(max(r0["elapsed"], r1["elapsed"]))
    assert r1["elapsed"] > r0["elapsed"]


def test_reference_arm_two_ranks_prints_once(tmp_path):
    """Under torchrun-style env, only rank 0 runs and prints the oracle line; rank 1 exits 0."""
    outs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
        p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                            "--workload", "tiny", "--steps", "3", "--warmup", "3"],
                           env=env, capture_output=True, text=True, timeout=300)
        assert p.returncode == 0, p.stderr
        outs.append(p.stdout.strip())
    line = json.loads(outs[0])
    assert outs[1] == ""
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    for k in ("metric", "value", "unit", "higher_is_better", "cpu_baseline", "e2e", "config"):
        assert k in line
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_accounting_k3():
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    cfg = workloads.config("k3")
    acct = bench.workload_accounting(cfg, workloads.lengths(cfg))
    assert acct["kv_bytes"] == 64 * 131072 * 1152                # 9.66 GB, the pages' 576 x 2 B per token
    assert acct["flops_alg"] == 64 * 131072 * 96 * 2176
