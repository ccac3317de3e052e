"""The N > 1 path of bench.py on CPU: replicas only (the GEMM does not
shard), so what runs across ranks is the launch through torch.distributed.run,
the barrier, the max / sum over ranks of the timing and the work, and the
reference arm's rank-0-only output.  gloo backend, world size 2, 127.0.0.1."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    ws, r, local = bench.dist_env()
    dist = bench.maybe_init_dist(ws, "gloo")
    bench.barrier(dist)
    res = {"ws": ws, "rank": r, "local": local,
           "max": bench.max_over_ranks(dist, 1.5 + r),
           "sum": bench.sum_over_ranks(dist, 10.0 * r + 1.0)}
    bench.barrier(dist)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, "rank%d.json" % rank), "w") as f:
        json.dump(res, f)


def test_rank_reductions_over_gloo(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for rank in range(2):
        res = json.load(open(tmp_path / ("rank%d.json" % rank)))
        assert res == {"ws": 2, "rank": rank, "local": rank, "max": 2.5, "sum": 12.0}


def test_single_process_helpers_are_identities():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.maybe_init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.25) == 3.25 and bench.sum_over_ranks(None, 7.0) == 7.0


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--cpu-budget", "0.5",
           "--workload", "fp16_1024_uniform"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "TFLOP/s"
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
