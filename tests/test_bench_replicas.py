"""The multi-rank host path of bench.py, on the CPU: dgrad runs as independent
replicas (one per GPU), so N > 1 adds only a gloo control group for the
barrier and the max-over-ranks timing; the reference arm runs on rank 0 alone.
"""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench = _bench()
    got = bench.max_over_ranks(10.0 + 5.0 * rank, world)  # rank 1 is the slower replica
    dist.barrier()
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_single_rank_is_identity():
    assert _bench().max_over_ranks(3.5, 1) == 3.5


def test_max_over_ranks_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    results = dict(q.get(timeout=5) for _ in range(2))
    assert results == {0: 15.0, 1: 15.0}


def test_reference_arm_under_torchrun_prints_once():
    """Two ranks under torchrun: rank 0 times the oracle and prints the one JSON
    line, rank 1 exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--ref-images", "1",
           "--layers", "L20_1x1_2048-512_7"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["config"]["layers"] == 1 and rec["n_gpus"] == 2
