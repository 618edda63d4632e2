"""The bench's N > 1 path on the host: two ranks over gloo on the CPU run bench.Replicas as the
GPU ranks do over NCCL (barrier, slowest-rank time, whole-job throughput), with no data-path
collective."""

import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(ws),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    got_ws, got_rank, _ = bench._dist()
    rep = bench.Replicas(got_ws, got_rank, "cpu", backend="gloo")
    rep.barrier()
    slowest = rep.max_over_ranks(10.0 + 5.0 * rank)          # rank r "took" 10 + 5 r ms
    value = rep.whole_job(4096, slowest)
    rep.barrier()
    rep.close()
    out.put((rank, slowest, value))


def test_two_replicas_over_gloo():
    ws = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, out)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # every rank sees the slowest rank's time and the same whole-job value: 2 x 4096 tokens in 15 ms
    assert [r[1] for r in res] == [15.0, 15.0]
    assert all(r[2] == pytest.approx(2 * 4096 / 0.015) for r in res)


def test_single_replica_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    rep = bench.Replicas(1, 0, "cpu")
    rep.barrier()
    assert rep.max_over_ranks(3.5) == 3.5
    assert rep.whole_job(100, 10.0) == pytest.approx(10000.0)
    assert not torch.distributed.is_initialized()
    rep.close()


def test_reference_arm_other_ranks_exit_quietly():
    """Under torchrun the reference arm runs on rank 0 alone: any other rank exits 0 at once and
    prints nothing."""
    import subprocess
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
