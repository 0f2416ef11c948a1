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


def test_roofline_record_fraction_and_fields():
    b = load_bench()
    rec = b.roofline_record("k", 967.05, 1934.1, "measured", "no-such-record", 1000)
    assert rec["frac"] == pytest.approx(0.5)
    assert rec["bound"] == "tensor" and rec["unit"] == "TFLOP/s"
    assert rec["traffic"] is None  # no capture recorded under that key
    assert rec["algorithmic_bytes"] == 1000


def test_recorded_traffic_follows_its_sources(tmp_path, monkeypatch):
    # a record is used only while the sources it was captured on are unchanged
    import hashlib
    import json
    b = load_bench()
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    (tmp_path / "profiles").mkdir()
    rec = {"k": {"source_files": ["k.cu"], "traffic_bytes_per_launch": 123,
                 "source_sha256": hashlib.sha256(b"kernel v1").hexdigest()}}
    (tmp_path / "profiles" / "roofline_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(b, "ROOT", str(tmp_path))
    assert b.recorded_traffic("k") == 123
    assert b.recorded_traffic("other") is None
    src.write_text("kernel v2")
    assert b.recorded_traffic("k") is None


def test_committed_traffic_records_name_existing_sources():
    import json
    path = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    recs = json.load(open(path))
    assert {"fwd_bf16_b1h32n16384d128", "bwd_bf16_b4h16n2048d64", "fwd_e4m3_b4h16n4096d128"} <= set(recs)
    for rec in recs.values():
        for f in rec["source_files"]:
            assert os.path.exists(os.path.join(ROOT, f)), f
        assert rec["traffic_bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
