"""bench.py's host logic on CPU: two gloo ranks, each with its own step time,
must agree on the slowest one; the reference arm runs on rank 0 only and the
other ranks exit without work; the traffic key and the CPU description."""

import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(1.5 + rank * 0.75, world)
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29000 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 2.25, 1: 2.25}


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_reference_arm_non_zero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def _bench():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    return bench


def test_traffic_key_ignores_comments_but_not_code():
    """The ncu traffic figures are keyed by a digest of the kernel sources' code:
    editing a comment keeps them, editing code drops them (the roofline's traffic
    then reads null until a new capture)."""
    bench = _bench()
    src = {"k.cu": "// note\nint f() { return 1; }  // trailing\n/* block */\n"}
    base = bench.csrc_digest(src)
    assert bench.csrc_digest({"k.cu": "// other words\nint f() { return 1; }\n"}) == base
    assert bench.csrc_digest({"k.cu": "int f() { return 2; }\n"}) != base
    assert bench.csrc_digest({"k.cu": src["k.cu"], "new.cu": "int g();\n"}) != base


def test_cpu_model_is_reported():
    bench = _bench()
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()


def test_roofline_fields():
    bench = _bench()
    # 1 TFLOP at 1000 TF/s = 1 ms; 1 GB at 1000 GB/s = 1 ms; measured 2 ms -> half
    r = bench.roofline_fields(1e12, 1e9, 2.0, 1000.0, 1000.0)
    assert abs(r["roofline_us"] - 1000.0) < 1e-6 and abs(r["roofline_frac"] - 0.5) < 1e-12
    assert abs(r["gbs"] - 500.0) < 1e-9
    # four times the bytes: the HBM term binds
    r = bench.roofline_fields(1e12, 4e9, 8.0, 1000.0, 1000.0)
    assert r["roofline_bound"] == "hbm" and abs(r["roofline_frac"] - 0.5) < 1e-12
    # no HBM figure: only the tensor term
    assert bench.roofline_fields(1e12, 4e9, 2.0, 1000.0, 0.0)["roofline_bound"] == "tensor"
