"""The multi-process path of bench.py on CPU: two ranks over gloo (the GPU
runs use NCCL with the same calls).  Replicas only — no data-path
collective: the only exchanges are the barrier around the timed region and
the max over ranks of the timed milliseconds."""

import importlib.util
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    bench = _load_bench()
    w, r, _ = bench.dist_setup()
    bench.barrier(w)
    local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    total_ms = bench.max_over_ranks(local_ms, w)
    rate = bench.whole_job_rate(1000.0, total_ms, w)
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    out.put((r, w, total_ms, rate))


def test_two_ranks_max_time_and_whole_job_rate():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    results = [out.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    results.sort()
    assert [r for r, *_ in results] == [0, 1]
    for r, w, total_ms, rate in results:
        assert w == world
        assert total_ms == pytest.approx(15.0)  # the slowest rank's time on every rank
        assert rate == pytest.approx(2 * 1000.0 / 0.015)  # both ranks' work over that time


def test_single_rank_is_identity():
    bench = _load_bench()
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.whole_job_rate(10.0, 2000.0, 1) == pytest.approx(5.0)
