"""The multi-rank path on CPU (gloo, world size 2): the benchmark's
process-group setup, barrier and max-over-ranks timing, and the reference
arm launched by torch.distributed.run, where rank 0 alone works and prints
one JSON line and the other rank exits cleanly.  (The path shards as
independent replicas: no data-path collective exists to test.)"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, outdir):
    sys.path.insert(0, ROOT)
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": "2", "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    import torch.distributed as dist
    world, r, _ = bench.dist_setup(None)
    assert dist.get_backend() == "gloo"
    bench.barrier(world)
    v = bench.max_over_ranks(1.5 + r, world)  # rank 0: 1.5, rank 1: 2.5
    with open(os.path.join(outdir, "rank%d.json" % r), "w") as f:
        json.dump({"world": world, "rank": r, "max": v}, f)
    dist.destroy_process_group()


def test_max_over_ranks_gloo(tmp_path):
    if torch.cuda.is_available():
        pytest.skip("covers the CPU (gloo) process group")
    import torch.multiprocessing as mp
    mp.spawn(_rank_main, args=(free_port(), str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        with open(tmp_path / ("rank%d.json" % r)) as f:
            d = json.load(f)
        assert d == {"world": 2, "rank": r, "max": 2.5}


def test_reference_arm_two_ranks():
    if torch.cuda.is_available():
        pytest.skip("covers the CPU (gloo) launch")
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", PYTHONPATH=ROOT)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0", "--sample-stride", "4096"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    # the line carries every key of the benchmark contract
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["steps"] == 1 and d["warmup"] == 0 and d["higher_is_better"] is True
    assert d["unit"] == "GB/s" and d["ms_per_step"] > 0 and "workload" in d["config"]
    for k in ("value", "unit", "cores", "kind", "sample"):
        assert k in d["cpu_baseline"], k
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["cores"] >= 1
    for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert k in d["e2e"], k
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["unit"] == d["unit"]
