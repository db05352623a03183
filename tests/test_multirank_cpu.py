"""The bench's multi-rank path on CPU (gloo, world size 2).  The layer has no
cross-GPU step, so N > 1 runs N independent replicas: each rank times its
own layer, the ranks agree on the slowest time (the whole-job value divides
all ranks' tokens by it), and the reference arm runs on rank 0 alone.  No GPU
is used."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench
    w, r, _ = bench.dist_init()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    slowest = bench.max_over_ranks(1.5 * (rank + 1), w)   # rank 1 is the slow one
    with open(os.path.join(out_dir, "rank%d.txt" % rank), "w") as f:
        f.write(repr(slowest))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_ranks_agree_on_the_slowest_time(tmp_path):
    """Each rank passes its own time; both get the maximum back."""
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = [float((tmp_path / ("rank%d.txt" % r)).read_text()) for r in range(2)]
    assert got == [3.0, 3.0]


def _check_reference_line(res):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "gpu_launches"):
        assert key in res, key
    assert res["impl"] == "reference"
    assert res["value"] > 0 and res["unit"] == "tokens/s"
    assert res["cpu_baseline"]["kind"] == "oracle" and res["cpu_baseline"]["cores"] >= 1
    assert res["cpu_baseline"]["value"] == res["value"]
    assert res["e2e"] == {"value": res["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny_fp32", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    res = json.loads(lines[0])
    _check_reference_line(res)
    assert res["n_gpus"] == 1 and res["steps"] == 2 and res["config"]["workload"] == "tiny_fp32"


def test_reference_arm_under_two_ranks_prints_once():
    """torchrun with two ranks: rank 0 alone runs the oracle and prints; the
    other rank exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny_fp32",
           "--steps", "1", "--warmup", "1", "--gpus", "2"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    res = json.loads(lines[0])
    _check_reference_line(res)
    assert res["n_gpus"] == 2
