"""Host-side logic of bench.py on CPU: FLOP counting, whole-job throughput, and
the max-over-ranks timing reduction across a 2-process gloo group (the same
reduction the multi-GPU replica run uses over NCCL)."""
import importlib.util
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_flop_counts_follow_the_convention():
    b = load_bench()
    assert b.flops("fwd", 1, 32, 16384, 128, False) == 4 * 32 * 16384 ** 2 * 128
    assert b.flops("fwd", 1, 32, 16384, 128, True) == 2 * 32 * 16384 ** 2 * 128
    assert b.flops("fwdbwd", 4, 16, 2048, 64, False) == 14 * 64 * 2048 ** 2 * 64
    assert b.flops("fwd8", 4, 16, 4096, 128, False) == 4 * 64 * 4096 ** 2 * 128


def test_job_throughput_is_weak_scaling_aggregate():
    b = load_bench()
    assert b.job_tflops(1, 1e12, 1000.0) == pytest.approx(1.0)
    assert b.job_tflops(8, 1e12, 1000.0) == pytest.approx(8.0)


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    b = load_bench()
    # rank r reports step time 10 + r and e2e time 20 - r
    out = b.max_over_ranks([10.0 + rank, 20.0 - rank])
    dist.destroy_process_group()
    q.put((rank, out))


def test_max_over_ranks_with_gloo_world_2():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results[0] == results[1] == [11.0, 20.0]


def test_single_process_reduction_is_identity():
    b = load_bench()
    assert b.max_over_ranks([3.0, 4.0]) == [3.0, 4.0]
