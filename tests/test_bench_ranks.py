"""Host logic of the multi-process bench on CPU ranks (gloo, world size 2).

Every rank runs one replica of the step; the line reports the slowest rank's
step time and the units all ranks processed over it. No GPU is involved: the
rank reduction is the same call the bench makes, on gloo instead of NCCL.
"""
import importlib.util
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        # rank r measured (1.5 + r) ms per step; only rank 1 measured an e2e time
        got = b.max_over_ranks([1.5 + rank, 7.25 if rank == 1 else None, None], dist)
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks hold the slowest rank's step time; a value no rank measured stays None
    assert res[0] == res[1] == [2.5, 7.25, None]


def test_single_rank_values_unchanged():
    b = _bench()
    assert b.max_over_ranks([3.0, None], None) == [3.0, None]


def test_job_throughput_counts_every_replica():
    b = _bench()
    # 1 GB per step in 1 ms on one rank: 1000 GB/s; two replicas in the same time: twice that
    assert b.job_throughput(1, 1e9, 1.0, "GB/s") == pytest.approx(1000.0)
    assert b.job_throughput(2, 1e9, 1.0, "GB/s") == pytest.approx(2000.0)
    # 1e12 valid-tap FMAs in 100 ms: 20 TFLOP/s per replica
    assert b.job_throughput(1, 1e12, 100.0, "TFLOP/s") == pytest.approx(20.0)
    assert b.job_throughput(4, 1e12, 100.0, "TFLOP/s") == pytest.approx(80.0)


def test_reference_arm_other_ranks_exit_silently():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
