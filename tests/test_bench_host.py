"""Host logic of bench.py: the max-over-ranks timing reduction with two gloo ranks on CPU,
and the algorithmic FLOP / byte models against the layer definition."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench
from moe_inputs import configs


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, _ = bench.dist_info()
    bench.barrier(w)
    got = bench.max_over_ranks(10.0 + 5.0 * r, w)
    q.put((r, w, got))
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert res == [(0, 2, 15.0), (1, 2, 15.0)]


def test_flop_model_matches_definition():
    c = configs.CONFIGS[2]
    T, d, E, k, F, Fs = 8192, 7168, 256, 8, 2048, 2048
    assert bench.layer_flops(c) == T * (2 * d * E + k * 3 * 2 * d * F + 3 * 2 * d * Fs)
    assert abs(bench.layer_flops(c) / 1e12 - 6.524) < 0.001
    assert bench.gateup_flops(c) == 2 * d * (T * k + T) * 2 * F


def test_byte_model_counts_only_touched_experts():
    c = configs.CONFIGS[3]
    counts = np.zeros(256, dtype=np.int32)
    counts[:10] = 1
    s = 2
    want = 2 * 128 * 7168 * s + 256 * 7168 * s + 10 * 3 * 7168 * 2048 * s + 3 * 7168 * 2048 * s
    assert bench.layer_bytes(c, counts) == want


def test_code_digest_ignores_comments_but_not_code(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("// header\n__global__ void k(int* p) {\n  p[0] = 1;  /* store */\n}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    a = bench.code_digest(["k.cu"])
    src.write_text("// another header\n\n__global__ void k(int* p) {\n  p[0] = 1;\n}\n// end\n")
    assert bench.code_digest(["k.cu"]) == a
    src.write_text("__global__ void k(int* p) {\n  p[0] = 2;\n}\n")
    assert bench.code_digest(["k.cu"]) != a



def test_clock_summary_keeps_the_timed_region_only():
    """The clock record summarises only the nvidia-smi samples taken inside the timed region
    (with 50 ms of slack): idle samples around it, at the maximum clock, do not dilute the
    clock the timed passes ran at, and the throttle reasons seen inside are listed."""
    import time as _time
    base = _time.mktime(_time.strptime("2026/01/02 03:04:05", "%Y/%m/%d %H:%M:%S"))

    def line(dt, mhz, cap):
        t = base + dt
        stamp = _time.strftime("%Y/%m/%d %H:%M:%S", _time.localtime(int(t)))
        stamp += f".{int(round((t - int(t)) * 1000)):03d}"
        act = "Active" if cap else "Not Active"
        return (f"{stamp}, 0, {mhz}, 2032, 700.0, 0x0, Not Active, Not Active, Not Active, {act}")

    s = bench.ClockSampler(0)
    s.lines = [line(0.0, 2032, False), line(0.5, 2032, False),          # idle before
               line(1.00, 1450, True), line(1.05, 1470, True), line(1.10, 1460, True),
               line(1.60, 2032, False), line(2.0, 2032, False)]          # idle after
    out = s.summary(base + 1.0, base + 1.1)
    assert out["samples"] == 3
    assert out["sm_mhz"] == 1460.0 and out["sm_max_mhz"] == 2032.0
    assert out["reasons"] == ["sw_power_cap"] and out["sw_power_cap_samples"] == 3
    # a region shorter than the sampling period falls back to the nearest samples, and says so
    out = s.summary(base + 1.3, base + 1.32)
    assert "note" in out and out["samples"] == 3
