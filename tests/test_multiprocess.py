"""The N > 1 path of bench.py on the CPU: replicas only (the convolution has no exchange step), so
ranks meet at a barrier and in the maximum of their timed durations; under torchrun the CPU oracle
arm runs on rank 0 alone and the other ranks exit 0 without output. World size 2, gloo backend,
rendezvous on 127.0.0.1."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist("gloo")
    assert d.world == world and d.rank == rank and d.on
    d.barrier()
    # every rank reports its own step time; the job's time is the slowest rank's
    out[rank] = d.max(10.0 + 3.5 * rank)
    d.barrier()
    d.close()


def test_dist_max_over_two_gloo_ranks():
    port = _free_port()
    # the manager's server process starts by spawn: earlier tests may have left threads running
    # in this process, and a fork taken while another thread holds a lock can hang the child
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
        assert dict(out) == {0: 13.5, 1: 13.5}


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    env = {k: os.environ.pop(k) for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK") if k in os.environ}
    try:
        d = bench.Dist("gloo")
        assert d.world == 1 and not d.on and d.max(4.0) == 4.0
    finally:
        os.environ.update(env)


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3", "--config", "0",
           "--ref-seconds", "2"]
    r = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
