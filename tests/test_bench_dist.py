"""bench.py's multi-process path on CPU: two gloo ranks on 127.0.0.1.

Each rank runs its own replica (weak scaling, no data-path collective); the
only collectives are the timing barrier and the max/sum reductions, checked
here; and the reference arm under torchrun prints from rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    d = bench.init_dist(world, "gloo")
    mx = bench.max_over_ranks(d, float(rank + 1) * 10.0)
    sm = bench.sum_over_ranks(d, float(rank + 1))
    d.barrier()
    out[rank] = (mx, sm)
    dist.destroy_process_group()


def test_max_and_sum_over_two_ranks():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        assert out[0] == (20.0, 3.0) and out[1] == (20.0, 3.0)


def test_single_process_helpers_are_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 3.5) == 3.5
    assert bench.sum_over_ranks(None, 2.0) == 2.0


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "1",
           "--ref-seconds", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"


def _run_reference(extra):
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--steps", "2", "--warmup", "1", "--ref-seconds", "1"] + extra
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_backward_reference_arm_under_torchrun_prints_once():
    rec = _run_reference(["--op", "bwd", "--workload", "tiny"])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["metric"].startswith("attention bwd") and rec["unit"] == "TFLOP/s"
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["e2e"]["d2h_bytes_per_step"] == 0


def test_decode_reference_arm_under_torchrun_prints_once():
    rec = _run_reference(["--op", "decode", "--workload", "decode_small"])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["metric"].startswith("decoding attention") and rec["unit"] == "GB/s"
    assert rec["config"]["Nq"] == 2 and rec["config"]["Nk"] == 1024
    # a K/V cache this small (1 MB) sits in L2: its steps are timed after a flush
    assert rec["config"]["l2"].startswith("flushed")
