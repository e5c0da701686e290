#!/usr/bin/env python
"""Benchmark of the local MoE layer of one expert-parallel rank on GB300.

One step = one pass of the whole hot path over one batch of seeded synthetic
input: route -> dispatch -> gate/up GEMM + SwiGLU -> down GEMM -> combine, as
one moe_layer call through the C ABI (its split kernels for prefill-sized
workloads, its single fused launch for decode-sized ones, T*k <=
MOE_FUSED_MAX_PAIRS).  For the split path a second loop calls the step's
entries one by one (moe_route, moe_dispatch, moe_expert_gate_up,
moe_expert_down, moe_combine) with CUDA events between them, for the per-kernel
breakdown and the roofline of the two grouped GEMMs.  Inputs are resident in
HBM; L2 is flushed (256 MiB write) between timed steps, outside the timed
region.  After the timed region the same step runs back to back for a few
seconds under a 100 ms nvidia-smi sampler, so that the clock record describes
the kernels under load (the timed region itself lasts milliseconds).

Prints one JSON line.  `value` is routed tokens/s (T / step time, summed over
replicas for N > 1: every rank runs its own replica, no collective on the data
path).  `e2e` is the same metric through moe_layer with host buffers: pinned
host->device copies of x and logits and the device->host copy of the output
inside the timed region.  `--impl reference` times the CPU oracle instead.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer routed tokens/s + TFLOP/s (prefill), weight GB/s (decode), 1 GB300"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
NOMINAL_BF16_DENSE_TFLOPS = 2250.0  # GB300 dense bf16 tensor peak, vendor figure
NOMINAL_FP8_DENSE_TFLOPS = 4500.0  # GB300 dense fp8 tensor peak, vendor figure
LOAD_SECONDS = 3.0  # back-to-back steps under the clock sampler, outside the timed events
L2_FLUSH_BYTES = 256 << 20
_CS = "expert_routing_dispatch_gb300/csrc/"
KERNEL_SOURCES = {
    "grouped_gemm_gate_up": [_CS + "grouped_ffn.cu", _CS + "grouped_gemm_pair.cuh", _CS + "common.cuh"],
    "grouped_gemm_down": [_CS + "grouped_ffn.cu", _CS + "grouped_gemm_pair.cuh", _CS + "common.cuh"],
    "grouped_ffn_mx": [_CS + "mxfp8.cu", _CS + "grouped_gemm_mx.cuh", _CS + "common.cuh"],
    "moe_layer_fused": [_CS + "decode_fused.cu", _CS + "grouped_gemm.cuh", _CS + "common.cuh", _CS + "route.cuh",
                        _CS + "combine.cuh"],
    "moe_layer_mx_fused": [_CS + "mxfp8.cu", _CS + "grouped_gemm_mx.cuh", _CS + "common.cuh", _CS + "route.cuh",
                           _CS + "combine.cuh"],
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default="prefill_ep_rank")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--precision", choices=["bf16", "mxfp8"], default="bf16",
                   help="expert GEMM operands: bf16 (the workload's statement), or MXFP8 expert weights and "
                        "activations (moe_layer_mxfp8; weights quantised on the device before timing)")
    p.add_argument("--dispatch", choices=["copy", "gather"], default="copy",
                   help="copy: dispatch stages the token rows in x_perm (moe_layer); gather: the gate/up GEMM "
                        "gathers them from x by TMA (moe_layer_gather, decode-sized bf16 workloads only)")
    return p.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


def reduce_max(value, world, device=None):
    """Max of a per-rank time over all ranks (only the bench's bookkeeping uses a
    collective; the MoE data path has none)."""
    if world == 1:
        return float(value)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, tokens_per_rank, t_max_ms):
    """Whole-job tokens/s: every rank processes its own replica of the workload."""
    return world * tokens_per_rank / (t_max_ms * 1e-3)


def memory_bound_rates(T, E, k, H, R, t_local, kern_ms, hbm_gbs):
    """Algorithmic GB/s of the HBM-bound entries of the split path, from the entry-by-entry
    times (ms): routing reads the logits and writes k ids and weights per token; dispatch
    reads the topk ids (histogram and placement passes), the x rows of the tokens with a
    local slot, and writes the grouped rows with their indices; combine reads the fp32
    y_perm rows, the slot rows and weights, and writes the fp32 output rows."""
    b = {
        "route": T * E * 4 + T * k * 8,
        "dispatch": 2 * T * k * 4 + t_local * H * 2 + R * H * 2 + R * 4 + T * k * 4,
        "combine": R * H * 4 + T * k * 8 + T * H * 4,
    }
    out = {}
    for nm, by in b.items():
        ms = kern_ms.get(nm)
        if ms:
            gbs = by / (ms * 1e-3) / 1e9
            out[nm] = {"bytes": int(by), "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / hbm_gbs, 4)}
    return out


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"]))}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, bf16_tflops_sustained=1700.0), "fallback"


def kernel_hash(kernel):
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, config):
    """DRAM bytes per launch of `kernel` on `config` from the committed ncu summary,
    if it was taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}.{config}.md")
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    kv = {}
    for ln in lines:
        if ln.startswith("- ") and ":" in ln:
            k, v = ln[2:].split(":", 1)
            kv[k.strip()] = v.strip().strip("`")
    try:
        if kv.get("kernel_source_sha256_16") != kernel_hash(kernel):
            return None
        return float(kv["dram_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


def sum_or_none(*vals):
    return None if any(v is None for v in vals) else float(sum(vals))


class ClockSampler:
    """nvidia-smi samples (every `period_ms`) while the block runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, period_ms=200):
        self.gpu = gpu_index
        self.period_ms = period_ms
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def rows(self):
        rows = []
        for ln in (self.out or "").splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), max=float(f[2]), power=float(f[3]), hw=f[5], hwt=f[6], swt=f[7],
                                 pcap=f[8]))
            except ValueError:
                continue
        return rows

    def summary(self, loaded_w=200.0):
        """Median SM clock of the samples drawing more than `loaded_w` watts (all
        samples if none does), the maximum clock, and every throttle reason seen."""
        rows = self.rows()
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [r for r in rows if r["power"] > loaded_w]
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                              ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        use = loaded or rows
        return {"sm_mhz": statistics.median(r["sm"] for r in use), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_median_under_load": statistics.median(r["power"] for r in use),
                "power_w_max": max(r["power"] for r in rows)}


def clocks_record(timed, load, load_s, load_steps, kern_ms, dominant):
    """The JSON line's clock record: the median SM clock of the samples taken while
    the same step ran back to back for `load_s` seconds (the timed region itself is
    too short for the 100-200 ms sampler), every throttle reason seen in either
    window, and each dominant kernel's event time x that clock (kilocycles)."""
    lt, tt = load.summary(loaded_w=400.0), timed.summary()
    rec = dict(lt)
    rec["reasons"] = sorted(set(lt.get("reasons", [])) | set(tt.get("reasons", [])) - {"no samples"})
    rec["source"] = (f"nvidia-smi every {load.period_ms} ms while {load_steps} steps ran back to back for "
                     f"{load_s:.1f} s after the timed region; samples above 400 W count as under load")
    rec["timed_region"] = tt
    if lt.get("sm_mhz"):
        rec["kcycles_at_median_clock"] = {nm: round(kern_ms[nm] * lt["sm_mhz"], 1) for nm in dominant
                                          if kern_ms.get(nm)}
    return rec


def cpu_baseline(cfg, inp, seconds, gpu_out=None):
    """The oracle as it stands, on a bounded sample of the workload's tokens, in
    two phases: route + dispatch over all T tokens, and the token-major layer
    (its FFN + combine dominate) on the sample.  With `gpu_out` (the GPU's layer
    output, host array [T, H]) the sampled tokens also give the accuracy figure
    max |gpu - oracle| / RMS(oracle)."""
    import numpy as np

    import oracle

    T, k, e0, e1 = cfg["T"], cfg["k"], cfg["e0"], cfg["e1"]
    t0 = time.perf_counter()
    st, idx, _ = oracle.route(inp["logits"], k)
    assert st == 0
    oracle.dispatch(idx, e0, e1)
    t_rd = time.perf_counter() - t0

    def run(ntok, start):
        toks = (np.arange(ntok, dtype=np.int64) + start) % T
        t0 = time.perf_counter()
        st, ref = oracle.moe_layer_tokens(inp["logits"], inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"], k, e0,
                                          e1, tokens=toks)
        assert st == 0
        return time.perf_counter() - t0, toks, ref

    probe = min(T, 64)
    dt, _, _ = run(probe, 0)
    n = int(min(T, max(probe, probe * seconds / max(dt, 1e-6))))
    dt, toks, ref = run(n, probe)
    out = {"value": n / dt, "unit": "tokens/s", "cores": oracle.num_threads(), "nproc": os.cpu_count(),
           "kind": "oracle",
           "sample": f"{n} of {T} tokens (route + SwiGLU FFN of their local slots + combine, token-major, fp64)",
           "seconds": round(dt, 2),
           "phases": {"route_dispatch": {"tokens": T, "seconds": round(t_rd, 4), "tokens_per_s": T / t_rd},
                      "ffn_combine": {"tokens": n, "seconds": round(dt, 2), "tokens_per_s": n / dt,
                                      "note": "oracle_moe_layer_tokens on the sample; its per-token routing is "
                                              "under 0.1% of it"}}}
    if gpu_out is not None:
        rms = float(np.sqrt(np.mean(ref ** 2)))
        err = float(np.abs(gpu_out[toks].astype(np.float64) - ref).max())
        out["max_err_over_rms"] = err / rms if rms > 0 else err
        out["accuracy_tokens"] = int(toks.size)
    return out


def run_reference(args):
    """The CPU oracle timed as the reference arm (rank 0 only)."""
    rank, _, world = dist_env()
    if rank != 0:
        return
    import numpy as np

    import oracle
    import synth

    cfg = synth.config(args.config)
    inp = synth.make_inputs(cfg)
    T, k, e0, e1 = cfg["T"], cfg["k"], cfg["e0"], cfg["e1"]
    per_step = min(T, 128)
    times = []
    for i in range(args.warmup + args.steps):
        toks = (np.arange(per_step, dtype=np.int64) + i * per_step) % T
        t0 = time.perf_counter()
        st, _ = oracle.moe_layer_tokens(inp["logits"], inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"], k, e0, e1,
                                        tokens=toks)
        assert st == 0
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    t = sum(times) / len(times)
    value = per_step / t
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": workload_config(cfg, None),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"{per_step} tokens per step of the {cfg['name']} workload"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(cfg, R):
    T, H, I, E, k, e0, e1 = (cfg[n] for n in ("T", "H", "I", "E", "k", "e0", "e1"))
    c = {"workload": f"{cfg['name']}: T={T} H={H} I={I} E={E} top-{k}, local experts [{e0},{e1})",
         "T": T, "H": H, "I": I, "E": E, "k": k, "e0": e0, "e1": e1, "l2": "256 MiB L2 flush between timed steps"}
    if R is not None:
        c["R_routed_rows"] = R
    return c


def run_ours(args):
    import numpy as np
    import torch

    import expert_routing_dispatch_gb300 as moe
    import synth

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    moe.lib()

    cfg = synth.config(args.config)
    T, H, I, E, k, e0, e1 = synth.dims_of(cfg)
    n = e1 - e0
    P = T * k
    inp = synth.make_inputs(cfg)
    g = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)
    x, lg, wg, wu, wd = (g(inp[nm]) for nm in ("x", "logits", "w_gate", "w_up", "w_down"))
    dims = moe.Dims(T, H, I, E, k, e0, e1)
    i32, f32 = torch.int32, torch.float32
    topk_idx = torch.empty((T, k), dtype=i32, device=dev)
    topk_w = torch.empty((T, k), dtype=f32, device=dev)
    counts = torch.empty(n, dtype=i32, device=dev)
    offsets = torch.empty(n + 1, dtype=i32, device=dev)
    row_pair = torch.empty(P, dtype=i32, device=dev)
    pair_row = torch.empty(P, dtype=i32, device=dev)
    x_perm = torch.empty((P, H), dtype=torch.int16, device=dev)
    h = torch.empty((P, 2 * I), dtype=torch.int16, device=dev)  # bf16 hi and lo terms of h
    y_perm = torch.empty((P, H), dtype=f32, device=dev)
    out = torch.empty((T, H), dtype=f32, device=dev)
    status = torch.zeros(1, dtype=i32, device=dev)
    dws = moe.alloc_workspace(moe.moe_dispatch_workspace_size(dims), dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    mx = args.precision == "mxfp8"
    if mx:
        # MXFP8 expert weights, quantised once on the device (outside every timed region)
        u8 = torch.uint8
        wq = {}
        for key, w_, rows_, K_ in (("g", wg, n * I, H), ("u", wu, n * I, H), ("d", wd, n * H, I)):
            q_ = torch.empty((rows_, K_), dtype=u8, device=dev)
            s_ = torch.empty((rows_, K_ // 32), dtype=u8, device=dev)
            moe.moe_quantize_mxfp8(w_, rows_, K_, q_, s_, stream=sh)
            wq[key] = (q_, s_)
        torch.cuda.synchronize()
        lws = moe.alloc_workspace(moe.moe_layer_mxfp8_workspace_size(dims), dev)
    else:
        lws = moe.alloc_workspace(moe.moe_workspace_size(dims), dev)

    gather = args.dispatch == "gather"
    if gather and (mx or P > moe.FUSED_MAX_PAIRS):
        raise SystemExit("--dispatch gather: bf16 decode-sized workloads only (T*k <= %d)" % moe.FUSED_MAX_PAIRS)
    layer_fn = moe.moe_layer_gather if gather else moe.moe_layer

    def run_layer(x_, lg_, out_, **kw):
        if mx:
            moe.moe_layer_mxfp8(dims, x_, lg_, wq["g"], wq["u"], wq["d"], out_, lws, status=status, stream=sh, **kw)
        else:
            layer_fn(dims, x_, lg_, wg, wu, wd, out_, lws, status=status, stream=sh, **kw)

    fused = P <= moe.FUSED_MAX_PAIRS and not mx
    mx_fused = P <= moe.FUSED_MAX_PAIRS and mx
    # the timed step: one moe_layer call (decode-sized: one persistent launch; else
    # route + dispatch place/gather + gate/up + down + combine)
    names = ["layer_fused" if fused else "layer_mxfp8" if mx else "layer"]
    # route, place, row copy (for MXFP8: quantised once per token), gate/up, down, combine
    launches_per_step = 1 if fused or mx_fused else 6

    def step(evs):
        evs[0].record(stream)
        run_layer(x, lg, out, topk_idx=topk_idx, topk_w=topk_w)
        evs[1].record(stream)

    if not fused and not mx:
        # breakdown loop (not the headline): the same work as separate entry calls
        bnames = ["route", "dispatch", "gate_up", "down", "combine"]

        def bstep(evs):
            evs[0].record(stream)
            moe.moe_route(dims, lg, topk_idx, topk_w, status, stream=sh)
            evs[1].record(stream)
            moe.moe_dispatch(dims, x, topk_idx, counts, offsets, row_pair, pair_row, x_perm, dws, stream=sh)
            evs[2].record(stream)
            moe.moe_expert_gate_up(dims, x_perm, offsets, wg, wu, h, status, stream=sh)
            evs[3].record(stream)
            moe.moe_expert_down(dims, h, offsets, wd, y_perm, status, stream=sh)
            evs[4].record(stream)
            moe.moe_combine(dims, y_perm, pair_row, topk_w, out, stream=sh)
            evs[5].record(stream)

    mk = lambda k=len(names): [torch.cuda.Event(enable_timing=True) for _ in range(k + 1)]
    for _ in range(args.warmup):
        flush.zero_()
        step(mk())
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    all_evs = []
    wall0 = time.perf_counter()
    with ClockSampler(local_rank) as clk:
        for _ in range(args.steps):
            flush.zero_()  # outside the event bracket
            evs = mk()
            step(evs)
            all_evs.append(evs)
        torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    step_ms = [evs[0].elapsed_time(evs[-1]) for evs in all_evs]
    t_step = sum(step_ms) / len(step_ms)
    kern_ms = {names[0]: t_step}
    if mx:
        # the MXFP8 expert FFN alone (both GEMMs, moe_expert_ffn_mxfp8) on this run's grouped rows
        moe.moe_route(dims, lg, topk_idx, topk_w, status, stream=sh)
        moe.moe_dispatch(dims, x, topk_idx, counts, offsets, row_pair, pair_row, x_perm, dws, stream=sh)
        xpq = torch.empty((P, H), dtype=torch.uint8, device=dev)
        xps = torch.empty((P, H // 32), dtype=torch.uint8, device=dev)
        moe.moe_quantize_mxfp8(x_perm, P, H, xpq, xps, stream=sh)
        fws = moe.alloc_workspace(moe.moe_expert_ffn_mxfp8_workspace_size(dims), dev)
        ts = []
        for i in range(args.warmup + args.steps):
            flush.zero_()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            moe.moe_expert_ffn_mxfp8(dims, xpq, xps, offsets, wq["g"], wq["u"], wq["d"], y_perm, fws, status=status,
                                     stream=sh)
            a1.record(stream)
            a1.synchronize()
            if i >= args.warmup:
                ts.append(a0.elapsed_time(a1))
        kern_ms["ffn_mxfp8"] = sum(ts) / len(ts)
        assert int(status.item()) == 0, f"device status {int(status.item())}"
    if not fused and not mx:
        # per-kernel breakdown from the entry-by-entry loop (same warm-up, flush and step count)
        b_evs = []
        for i in range(args.warmup + args.steps):
            flush.zero_()
            evs = mk(len(bnames))
            bstep(evs)
            if i >= args.warmup:
                b_evs.append(evs)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"device status {int(status.item())}"
        for i, nm in enumerate(bnames):
            kern_ms[nm] = sum(e[i].elapsed_time(e[i + 1]) for e in b_evs) / len(b_evs)
        kern_ms["entries_total"] = sum(e[0].elapsed_time(e[-1]) for e in b_evs) / len(b_evs)
    # clock under load: the same step back to back (no flush) with the sampler at
    # 100 ms, outside the timed events, so the clock record describes the kernels
    torch.cuda.synchronize()
    load_steps = 0
    with ClockSampler(local_rank, period_ms=100) as clk_load:
        t_load0 = time.perf_counter()
        while time.perf_counter() - t_load0 < LOAD_SECONDS:
            for _ in range(20):
                run_layer(x, lg, out, topk_idx=topk_idx, topk_w=topk_w)
            load_steps += 20
            torch.cuda.synchronize()
        t_load = time.perf_counter() - t_load0
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    out_for_accuracy = None if mx else out.cpu().numpy()  # the bf16 oracle is the reference of the bf16 path
    # routed rows and active local experts, counted from this run's routing
    ti = topk_idx.flatten()
    loc = ti[(ti >= e0) & (ti < e1)]
    t_local = int(((topk_idx.view(T, k) >= e0) & (topk_idx.view(T, k) < e1)).any(dim=1).sum().item())
    R = int(loc.numel())
    active = int(torch.unique(loc).numel())
    t_step_max = reduce_max(t_step, world, dev)

    # ---- end to end through moe_layer with host buffers
    # Every step uploads its x and logits from pinned host memory, runs moe_layer
    # and downloads the fp32 output.  Serving-style pipeline: uploads, layers and
    # downloads of consecutive steps run on three streams with double-buffered
    # device tensors, so step i+1's upload and step i-1's download overlap step
    # i's layer.  The per-step serial figure (copies and layer back to back,
    # L2 flushed before each step) is reported beside it.
    x_h = torch.from_numpy(inp["x"].view(np.int16)).pin_memory()
    lg_h = torch.from_numpy(inp["logits"]).pin_memory()
    out_h = [torch.empty((T, H), dtype=f32).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(x) for _ in range(2)]
    lg_d = [torch.empty_like(lg) for _ in range(2)]
    out_d = [torch.empty((T, H), dtype=f32, device=dev) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: [torch.cuda.Event() for _ in range(2)]
    ev_in, ev_comp, ev_out = ev(), ev(), ev()

    def serial_step():
        x_d[0].copy_(x_h, non_blocking=True)
        lg_d[0].copy_(lg_h, non_blocking=True)
        run_layer(x_d[0], lg_d[0], out_d[0])
        out_h[0].copy_(out_d[0], non_blocking=True)

    def pipelined(steps):
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        for i in range(steps):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[b])  # layer i-2 has read x_d[b], lg_d[b]
                x_d[b].copy_(x_h, non_blocking=True)
                lg_d[b].copy_(lg_h, non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])  # download i-2 has read out_d[b]
            run_layer(x_d[b], lg_d[b], out_d[b])
            ev_comp[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[b])
                out_h[b].copy_(out_d[b], non_blocking=True)
                ev_out[b].record(s_out)
        s_out.wait_event(ev_out[(steps - 1) % 2])
        t1.record(s_out)
        t1.synchronize()
        return t0.elapsed_time(t1) / steps

    for _ in range(max(1, args.warmup)):
        serial_step()
    torch.cuda.synchronize()
    serial_ms = []
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        serial_step()
        b.record(stream)
        b.synchronize()
        serial_ms.append(a.elapsed_time(b))
    t_e2e_serial = reduce_max(sum(serial_ms) / len(serial_ms), world, dev)
    pipelined(max(2, args.warmup))
    torch.cuda.synchronize()
    t_e2e = reduce_max(pipelined(args.steps), world, dev)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    flop_gate_up = 4.0 * H * I * R
    flop_layer = 6.0 * H * I * R
    # weight bytes streamed per step: bf16, or E4M3 codes plus one UE8M0 scale per 32
    weight_bytes = 3.0 * H * I * (1.0 + 1.0 / 32 if mx else 2.0) * active
    if fused:
        # HBM roofline of the fused launch: active experts' weights streamed once,
        # plus x, logits and the fp32 output (intermediates stay in L2)
        alg_bytes = weight_bytes + T * H * 2 + T * E * 4 + T * H * 4
        achieved = alg_bytes / (kern_ms["layer_fused"] * 1e-3) / 1e9
        roofline = {"kernel": "moe_layer_fused_kernel (route..combine, one cooperative launch)", "bound": "hbm",
                    "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": achieved / peaks["hbm_gbs"], "peak_source": f"{peak_src} HBM copy",
                    "traffic": recorded_traffic("moe_layer_fused", args.config),
                    "algorithmic_bytes_per_launch": alg_bytes}
    elif mx_fused:
        # HBM roofline of the fused MXFP8 launch: the active experts' E4M3 codes and block
        # scales streamed once, plus x, logits and the fp32 output
        alg_bytes = weight_bytes + T * H * 2 + T * E * 4 + T * H * 4
        achieved = alg_bytes / (kern_ms["layer_mxfp8"] * 1e-3) / 1e9
        roofline = {"kernel": "moe_layer_mx_fused_kernel (route..combine, MXFP8 GEMMs, one cooperative launch)",
                    "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": achieved / peaks["hbm_gbs"], "peak_source": f"{peak_src} HBM copy",
                    "traffic": recorded_traffic("moe_layer_mx_fused", args.config),
                    "algorithmic_bytes_per_launch": alg_bytes}
    elif mx:
        # both MXFP8 grouped GEMMs against the fp8 tensor peak: the measured bf16 peak x 2
        # (the nominal dense ratio, 4.5 / 2.25 PFLOP/s)
        fp8_peak = 2.0 * peaks["bf16_tflops"]
        achieved = flop_layer / (kern_ms["ffn_mxfp8"] * 1e-3) / 1e12 if R else 0.0
        roofline = {"kernel": "grouped_ffn_mx_kernel gate/up + down (tcgen05 kind::mxf8f6f4 block-scaled)",
                    "bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                    "frac": achieved / fp8_peak, "peak_source": f"{peak_src} bf16 burst x 2 (nominal fp8 ratio)",
                    "frac_of_nominal_dense": achieved / NOMINAL_FP8_DENSE_TFLOPS,
                    "nominal_dense_peak": NOMINAL_FP8_DENSE_TFLOPS,
                    "traffic": recorded_traffic("grouped_ffn_mx", args.config),
                    "algorithmic_flop_per_launch": flop_layer}
    else:
        # both grouped GEMMs (gate/up + SiLU*up, down) against the bf16 tensor peak; the
        # gate/up GEMM alone (the largest kernel) as a secondary figure
        t_gemms = kern_ms["gate_up"] + kern_ms["down"]
        achieved = flop_layer / (t_gemms * 1e-3) / 1e12 if R else 0.0
        gu = flop_gate_up / (kern_ms["gate_up"] * 1e-3) / 1e12 if R else 0.0
        dn = (flop_layer - flop_gate_up) / (kern_ms["down"] * 1e-3) / 1e12 if R else 0.0
        roofline = {"kernel": "grouped_ffn gate/up (tcgen05, SiLU*up epilogue) + down, summed event times",
                    "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": achieved / peaks["bf16_tflops"], "peak_source": f"{peak_src} bf16 burst (cuBLAS)",
                    "frac_of_nominal_dense": achieved / NOMINAL_BF16_DENSE_TFLOPS,
                    "nominal_dense_peak": NOMINAL_BF16_DENSE_TFLOPS,
                    "traffic": sum_or_none(recorded_traffic("grouped_gemm_gate_up", args.config),
                                           recorded_traffic("grouped_gemm_down", args.config)),
                    "traffic_note": "DRAM bytes of the gate/up and down launches (ncu), per step",
                    "algorithmic_bytes": (2 * H * I * 2 * active + R * H * 2 + R * 2 * I * 2) +
                                         (H * I * 2 * active + R * 2 * I * 2 + R * H * 4),
                    "algorithmic_flop_per_launch": flop_layer,
                    "gate_up": {"achieved": gu, "frac": gu / peaks["bf16_tflops"],
                                "frac_of_nominal_dense": gu / NOMINAL_BF16_DENSE_TFLOPS, "flop": flop_gate_up},
                    "down": {"achieved": dn, "frac": dn / peaks["bf16_tflops"],
                             "frac_of_nominal_dense": dn / NOMINAL_BF16_DENSE_TFLOPS,
                             "flop": flop_layer - flop_gate_up}}
    gemm_ms = (kern_ms["layer_fused"] if fused else kern_ms["ffn_mxfp8"] if mx else
               kern_ms["gate_up"] + kern_ms["down"])
    line = {
        "metric": METRIC,
        "value": job_throughput(world, T, t_step_max),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t_step_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "mxfp8 (e4m3, ue8m0 block-32 scales; fp32 accumulate)" if mx else "bf16",
        "data": "synthetic (seeded counter-based generator; random-init weights)",
        "config": dict(workload_config(cfg, R), **({"precision": "mxfp8"} if mx else {}),
                       **({"dispatch": "tma_row_gather"} if gather else {})),
        "e2e": {"value": job_throughput(world, T, t_e2e), "unit": "tokens/s",
                "h2d_bytes_per_step": int(inp["x"].nbytes + inp["logits"].nbytes),
                "d2h_bytes_per_step": int(T * H * 4),
                "ms_per_step": t_e2e,
                "serial_value": job_throughput(world, T, t_e2e_serial), "serial_ms_per_step": t_e2e_serial,
                "note": (("moe_layer_mxfp8" if mx else layer_fn.__name__) +
                         " per step with its pinned-host x/logits upload and fp32 output download; "
                         "value: uploads, layers and downloads of consecutive steps pipelined on 3 streams "
                         "(double-buffered); serial_value: copies and layer back to back, L2 flushed; "
                         "expert weights resident")},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": roofline,
        "clocks": clocks_record(clk, clk_load, t_load, load_steps, kern_ms,
                                [nm for nm in ("gate_up", "down", "layer", "layer_fused", "layer_mxfp8",
                                               "ffn_mxfp8") if nm in kern_ms]),
        "detail": {
            "kernel_ms": {nm: round(v, 4) for nm, v in kern_ms.items()},
            "layer_tflops": flop_layer / (t_step * 1e-3) / 1e12,
            "gemm_tflops": flop_layer / (gemm_ms * 1e-3) / 1e12,
            "path": "fused" if fused or mx_fused else "split",
            "active_local_experts": active,
            "routed_rows_per_s": R / (t_step * 1e-3),
            "weight_gbs": weight_bytes / (t_step * 1e-3) / 1e9,
            "memory_bound_entries": memory_bound_rates(T, E, k, H, int(loc.numel()), t_local, kern_ms,
                                                        peaks["hbm_gbs"]) if not fused and not mx else {},
            "wall_s_timed_loop_incl_flush": round(wall, 4),
            "step_ms_min": min(step_ms), "step_ms_max": max(step_ms),
        },
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, inp, args.cpu_seconds, gpu_out=out_for_accuracy)
        if "max_err_over_rms" in line["cpu_baseline"]:
            line["max_err_over_rms"] = line["cpu_baseline"]["max_err_over_rms"]
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
