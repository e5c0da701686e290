"""The multi-process (N > 1) bookkeeping of bench.py on CPU with gloo,
world_size 2: the timing max over ranks, the whole-job throughput of N
independent replicas, and the reference arm under torchrun (rank 0 alone
prints one line, the other rank exits 0 without work)."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [2.0, 3.5][rank]  # the slower rank sets the job's time
    t = bench.reduce_max(local_ms, world)
    q.put((rank, t, bench.job_throughput(world, 6000, t)))
    dist.destroy_process_group()


def test_reduce_max_and_job_throughput_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [3.5, 3.5]
    assert res[0][2] == pytest.approx(2 * 6000 / 3.5e-3)


def test_single_rank_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.reduce_max(1.25, 1) == 1.25
    assert bench.job_throughput(1, 256, 0.5) == pytest.approx(512000.0)


def test_reference_arm_under_torchrun_prints_once():
    port = 30500 + os.getpid() % 1000
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--config", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0


def test_memory_bound_rates_prefill_ep_rank_numbers():
    """The GB/s the JSON line reports for the HBM-bound entries: bytes counted per the
    stated formulas, rates from the entry times, fractions of the given HBM peak."""
    sys.path.insert(0, ROOT)
    import bench

    T, E, k, H, R, t_local = 6000, 128, 8, 4096, 12014, 5000
    r = bench.memory_bound_rates(T, E, k, H, R, t_local, {"route": 0.01, "combine": 0.0512}, 6796.9)
    assert set(r) == {"route", "combine"}  # no time for dispatch -> not reported
    assert r["route"]["bytes"] == 6000 * 128 * 4 + 6000 * 8 * 8 == 3_456_000
    assert abs(r["route"]["gbs"] - 345.6) < 0.05
    comb = 12014 * 4096 * 4 + 6000 * 8 * 8 + 6000 * 4096 * 4
    assert r["combine"]["bytes"] == comb == 295_525_376
    assert abs(r["combine"]["gbs"] - comb / 0.0512e-3 / 1e9) < 0.05
    assert abs(r["combine"]["frac_of_hbm"] - r["combine"]["gbs"] / 6796.9) < 1e-4
    d = bench.memory_bound_rates(T, E, k, H, R, t_local, {"dispatch": 0.0382}, 6796.9)["dispatch"]
    assert d["bytes"] == 2 * T * k * 4 + t_local * H * 2 + R * H * 2 + R * 4 + T * k * 4


def test_clock_record_uses_the_load_window():
    # fake nvidia-smi output: the timed region saw two idle samples, the load loop
    # six samples at dense-GEMM power and one idle; reasons from both windows count
    sys.path.insert(0, ROOT)
    import bench

    def sampler(lines, period):
        c = bench.ClockSampler(0, period_ms=period)
        c.out = "\n".join(lines)
        return c

    idle = "0, 2070, 2070, 180.5, 0x0, Not Active, Not Active, Not Active, Not Active"
    timed = sampler([idle, idle], 200)
    load = sampler([idle] + [f"0, {m}, 2070, {p}, 0x4, Not Active, Not Active, Not Active, Active"
                             for m, p in ((1650, 1390), (1700, 1380), (1680, 1395), (1720, 1370), (1690, 1385),
                                          (1710, 1388))], 100)
    rec = bench.clocks_record(timed, load, 3.0, 120, {"gate_up": 0.25, "down": 0.14}, ["gate_up", "down"])
    assert rec["samples_under_load"] == 6 and rec["sm_mhz"] == 1695.0
    assert rec["reasons"] == ["sw_power_cap"]
    assert rec["timed_region"]["samples"] == 2
    assert rec["kcycles_at_median_clock"] == {"gate_up": round(0.25 * 1695.0, 1), "down": round(0.14 * 1695.0, 1)}
