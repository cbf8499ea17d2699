"""Host logic of the benchmark's multi-GPU mode (independent replicas, no
data-path collective), run as two gloo ranks on the CPU: the timing is the
maximum over ranks and the whole-job rate counts the work of every rank."""
import importlib.util
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        bench = load_bench()
        assert bench.dist_env() == (ws, rank, rank)
        # rank r took 100 + 50 r ms for its 4 steps of 1e12 work units each
        rate, tmax = bench.whole_job_rate(100.0 + 50.0 * rank, ws, 1e12, 4)
        bench.barrier(ws)
        q.put((rank, rate, tmax))
    finally:
        dist.destroy_process_group()


def test_two_replicas_max_time_and_whole_job_rate():
    ws, port = 2, free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(ws))
    for rank, rate, tmax in got:
        assert tmax == pytest.approx(150.0)             # the slower rank's time
        assert rate == pytest.approx(2 * 1e12 * 4 / 0.150)  # both ranks' work


def test_single_rank_needs_no_process_group():
    bench = load_bench()
    rate, tmax = bench.whole_job_rate(200.0, 1, 5e11, 10)
    assert tmax == 200.0
    assert rate == pytest.approx(5e11 * 10 / 0.2)
