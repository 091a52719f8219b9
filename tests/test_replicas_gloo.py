"""Multi-rank plumbing of multi-GPU runs (replicas, no data-path collective), run as two gloo
ranks on the CPU: rendezvous on 127.0.0.1, barrier, maximum of the ranks' times, the whole-job
throughput, and that only rank 0 reports."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(r, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(r), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(r))
    from prefix_cached_kv_gb300 import replicas
    try:
        assert replicas.world() == world and replicas.rank() == r
        assert replicas.init("gloo") == "gloo"
        replicas.barrier()
        ms = 10.0 + 5.0 * r                       # rank r "took" 10 + 5 r ms
        mx = replicas.max_over_ranks(ms)
        value = replicas.job_throughput(1000.0, mx)
        replicas.barrier()
        out.put((r, mx, value, replicas.rank() == 0))
    finally:
        replicas.finish()


def test_two_gloo_ranks_agree_on_max_and_job_rate():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = [out.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    # both ranks see the slowest rank's time; the job rate counts both ranks' units over it
    for r, mx, value, reports in res:
        assert mx == 15.0
        assert value == pytest.approx(2 * 1000.0 / 15e-3)
        assert reports == (r == 0)


def test_single_process_is_a_one_rank_job(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    from prefix_cached_kv_gb300 import replicas
    assert replicas.world() == 1 and replicas.rank() == 0
    assert replicas.init() is None
    replicas.barrier()
    assert replicas.max_over_ranks(3.5) == 3.5
    assert replicas.job_throughput(10.0, 2.0) == pytest.approx(5000.0)
