"""Multi-process host logic of bench.py on CPU (gloo, world size 2): the
max-over-ranks reduction of the step time, and the reference arm under
torchrun (rank 0 alone prints one JSON line; the other ranks exit 0)."""

import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    # rank r measured 100 + 7 r microseconds per step
    got = bench.max_over_ranks(100.0 + 7.0 * rank, world, torch.device("cpu"))
    dist.barrier()
    out[rank] = got
    dist.destroy_process_group()


def test_step_time_is_the_max_over_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as man:
        out = man.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        assert dict(out) == {0: 107.0, 1: 107.0}


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, 1, None) == 12.5


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "c0", "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "us" and rec["value"] > 0
    assert rec["higher_is_better"] is False
    assert rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
