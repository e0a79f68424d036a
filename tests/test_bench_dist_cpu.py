"""The benchmark's multi-rank host logic on CPU (gloo, world size 2).

bench.py runs one process per GPU with no data exchange (independent
replicas): ranks meet only at the barriers around the timed region and in the
max-over-ranks reduction of the timings, and rank 0 alone prints.  These tests
run that logic on CPU ranks: the reduction and the barrier directly, and the
reference arm (the oracle on the host cores) end to end under torchrun.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
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
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cpu = torch.device("cpu")
        bench.barrier(dist, cpu)
        got = bench.max_over_ranks(dist, 1.5 + 2.0 * rank, cpu)
        bench.barrier(dist, cpu)
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        assert dict(out) == {0: 3.5, 1: 3.5}


def test_single_process_helpers_are_identities():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 2.25, torch.device("cpu")) == 2.25
    bench.barrier(None, torch.device("cpu"))


def test_reference_arm_under_torchrun_two_ranks():
    """Rank 0 runs the oracle and prints one JSON line; rank 1 exits 0 without
    output; both leave the process group cleanly."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "1", "--ref-tokens", "64"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["higher_is_better"] is True and d["config"]["workload"] == "gdn_prefill_bf16"
