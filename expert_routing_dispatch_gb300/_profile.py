"""Profiling drivers of the grouped GEMMs and of the layer, on one GPU.

    python -m expert_routing_dispatch_gb300._profile roles [workload ...]
        Where the grouped GEMMs' pipeline roles wait.  Builds a separate copy of
        libmoe with -DMOE_GEMM_PROFILE (every role of the bf16 CTA-pair GEMMs and
        of the MXFP8 GEMMs then sums the clock cycles it spends in its mbarrier
        waits), groups a workload's rows with moe_route + moe_dispatch, runs each
        GEMM three times as warm-up and then once more with L2 flushed between the
        counter reset and the read, and prints one markdown table row per GEMM:
        wait cycles / the role's cycles in the kernel.  For decode-sized workloads
        (T*k <= MOE_FUSED_MAX_PAIRS) the MXFP8 rows are the GEMM phases inside the
        fused moe_layer_mxfp8 launch.  The product library is
        untouched: the counters exist only in the copy built here
        (_lib/libmoe_prof.so).

    python -m expert_routing_dispatch_gb300._profile phases [workload ...]
        Where the fused single-launch layers (bf16 moe_layer and moe_layer_mxfp8 at
        T*k <= MOE_FUSED_MAX_PAIRS) spend their time.  The same profile copy of the
        library stamps %globaltimer in every CTA at each phase boundary (after a block
        barrier); per phase the table gives the time from the last CTA entering it to
        the last CTA leaving it (medians of 6 launches, L2 flushed before each).

    python -m expert_routing_dispatch_gb300._profile steps [--config W] [--warmup N] [--steps K] [--precision P]
        A short, fixed launch sequence of the product library for ncu: N + K
        moe_layer (or moe_layer_mxfp8) steps with a 256 MiB L2 flush before each,
        then one pass of the split entries (moe_route, moe_dispatch,
        moe_expert_gate_up, moe_expert_down, moe_combine).
"""
import ctypes
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
PROF_LIB = os.path.join(HERE, "_lib", "libmoe_prof.so")


def _frac(a, b):
    return a / b if b else 0.0


def measure(name):
    import numpy as np
    import torch

    import expert_routing_dispatch_gb300 as moe
    import synth

    cfg = synth.config(name)
    T, H, I, E, k, e0, e1 = synth.dims_of(cfg)
    n, P = e1 - e0, T * k
    inp = synth.make_inputs(cfg)
    dev = torch.device("cuda")
    g = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)
    x, lg, wg, wu, wd = (g(inp[nm]) for nm in ("x", "logits", "w_gate", "w_up", "w_down"))
    i32 = torch.int32
    idx, w = torch.empty((T, k), dtype=i32, device=dev), torch.empty((T, k), dtype=torch.float32, device=dev)
    counts, offsets = torch.empty(n, dtype=i32, device=dev), torch.empty(n + 1, dtype=i32, device=dev)
    row_pair, pair_row = torch.empty(P, dtype=i32, device=dev), torch.empty(P, dtype=i32, device=dev)
    x_perm = torch.empty((P, H), dtype=torch.int16, device=dev)
    h = torch.empty((P, 2 * I), dtype=torch.int16, device=dev)
    y = torch.empty((P, H), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=i32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    moe.moe_route(cfg, lg, idx, w, status)
    moe.moe_dispatch(cfg, x, idx, counts, offsets, row_pair, pair_row, x_perm,
                     moe.alloc_workspace(moe.moe_dispatch_workspace_size(cfg)))
    L = moe.lib()
    L.moe_debug_gemm_prof.argtypes = [ctypes.c_void_p, ctypes.c_int]
    L.moe_debug_mx_prof.argtypes = [ctypes.c_void_p, ctypes.c_int]
    rows = []

    def timed(launch, read, nctr):
        for _ in range(3):
            launch()
        torch.cuda.synchronize()
        flush.zero_()
        buf = (ctypes.c_ulonglong * nctr)()
        read(buf, 1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        launch()
        b.record()
        torch.cuda.synchronize()
        read(buf, 1)
        assert int(status.item()) == 0
        return a.elapsed_time(b), list(buf)

    # bf16 CTA-pair GEMMs: counters [0..7] gate/up, [8..15] down
    for mode, launch in (("gate/up", lambda: moe.moe_expert_gate_up(cfg, x_perm, offsets, wg, wu, h, status)),
                         ("down", lambda: moe.moe_expert_down(cfg, h, offsets, wd, y, status))):
        ms, c = timed(launch, L.moe_debug_gemm_prof, 16)
        c = c[:8] if mode == "gate/up" else c[8:]
        rows.append((f"bf16 {mode}", name, ms, c[7], _frac(c[3], c[4]), _frac(c[2], c[4]), _frac(c[0], c[1]),
                     _frac(c[5], c[6]), None))
    # MXFP8 FFN: [0..11] gate/up, [12..23] down (both GEMMs run in each launch)
    u8 = torch.uint8
    wq = {}
    for key, w_, r_, K_ in (("g", wg, n * I, H), ("u", wu, n * I, H), ("d", wd, n * H, I)):
        q_, s_ = torch.empty((r_, K_), dtype=u8, device=dev), torch.empty((r_, K_ // 32), dtype=u8, device=dev)
        moe.moe_quantize_mxfp8(w_, r_, K_, q_, s_)
        wq[key] = (q_, s_)
    xq, xs = torch.empty((P, H), dtype=u8, device=dev), torch.empty((P, H // 32), dtype=u8, device=dev)
    moe.moe_quantize_mxfp8(x_perm, P, H, xq, xs)
    fws = moe.alloc_workspace(moe.moe_expert_ffn_mxfp8_workspace_size(cfg))
    if P <= moe.FUSED_MAX_PAIRS:
        # decode sizes: the GEMM phases inside the fused moe_layer_mxfp8 launch
        lws = moe.alloc_workspace(moe.moe_layer_mxfp8_workspace_size(cfg))
        out = torch.empty((T, H), dtype=torch.float32, device=dev)
        launch, label = (lambda: moe.moe_layer_mxfp8(cfg, x, lg, wq["g"], wq["u"], wq["d"], out, lws,
                                                     status=status)), "mxfp8 fused"
    else:
        launch, label = (lambda: moe.moe_expert_ffn_mxfp8(cfg, xq, xs, offsets, wq["g"], wq["u"], wq["d"], y, fws,
                                                          status=status)), "mxfp8"
    ms, c = timed(launch, L.moe_debug_mx_prof, 24)
    for j, mode in enumerate(("gate/up", "down")):
        cc = c[12 * j:12 * j + 12]
        rows.append((f"{label} {mode}", name, ms, cc[10], _frac(cc[3], cc[5]), _frac(cc[2], cc[5]),
                     _frac(cc[0], cc[1]), _frac(cc[6], cc[7]), _frac(cc[8], cc[9])))
    return rows


def steps(argv):
    import argparse

    import numpy as np
    import torch

    import expert_routing_dispatch_gb300 as moe
    import synth

    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="prefill_ep_rank")
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--steps", type=int, default=1)
    ap.add_argument("--precision", choices=["bf16", "mxfp8"], default="bf16")
    a = ap.parse_args(argv)
    cfg = synth.config(a.config)
    T, H, I, E, k, e0, e1 = synth.dims_of(cfg)
    n, P = e1 - e0, T * k
    inp = synth.make_inputs(cfg)
    dev = torch.device("cuda")
    g = lambda x_: torch.from_numpy(x_.view(np.int16) if x_.dtype == np.uint16 else x_).to(dev)
    x, lg, wg, wu, wd = (g(inp[nm]) for nm in ("x", "logits", "w_gate", "w_up", "w_down"))
    out = torch.empty((T, H), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    if a.precision == "mxfp8":
        u8 = torch.uint8
        wq = {}
        for key, w_, r_, K_ in (("g", wg, n * I, H), ("u", wu, n * I, H), ("d", wd, n * H, I)):
            q_, s_ = torch.empty((r_, K_), dtype=u8, device=dev), torch.empty((r_, K_ // 32), dtype=u8, device=dev)
            moe.moe_quantize_mxfp8(w_, r_, K_, q_, s_)
            wq[key] = (q_, s_)
        ws = moe.alloc_workspace(moe.moe_layer_mxfp8_workspace_size(cfg))
        layer = lambda: moe.moe_layer_mxfp8(cfg, x, lg, wq["g"], wq["u"], wq["d"], out, ws, status=status)
    else:
        ws = moe.alloc_workspace(moe.moe_workspace_size(cfg))
        layer = lambda: moe.moe_layer(cfg, x, lg, wg, wu, wd, out, ws, status=status)
    for _ in range(a.warmup + a.steps):
        flush.zero_()
        layer()
    i32 = torch.int32
    idx, w = torch.empty((T, k), dtype=i32, device=dev), torch.empty((T, k), dtype=torch.float32, device=dev)
    counts, offsets = torch.empty(n, dtype=i32, device=dev), torch.empty(n + 1, dtype=i32, device=dev)
    row_pair, pair_row = torch.empty(P, dtype=i32, device=dev), torch.empty(P, dtype=i32, device=dev)
    x_perm = torch.empty((P, H), dtype=torch.int16, device=dev)
    h = torch.empty((P, 2 * I), dtype=torch.int16, device=dev)
    y = torch.empty((P, H), dtype=torch.float32, device=dev)
    flush.zero_()
    moe.moe_route(cfg, lg, idx, w, status)
    moe.moe_dispatch(cfg, x, idx, counts, offsets, row_pair, pair_row, x_perm,
                     moe.alloc_workspace(moe.moe_dispatch_workspace_size(cfg)))
    moe.moe_expert_gate_up(cfg, x_perm, offsets, wg, wu, h, status)
    moe.moe_expert_down(cfg, h, offsets, wd, y, status)
    moe.moe_combine(cfg, y, pair_row, w, out)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    print(f"steps ok: {a.config} {a.precision}: {a.warmup + a.steps} layer steps, then the split entries once")


PHASES = ("route", "barrier", "dispatch", "barrier", "gate/up GEMM", "barrier", "down GEMM", "barrier", "combine",
          "teardown")


def phases(argv):
    import statistics

    import numpy as np
    import torch

    import expert_routing_dispatch_gb300 as moe
    import synth
    from expert_routing_dispatch_gb300 import _build

    _build.build(force=True, extra_flags=["-DMOE_GEMM_PROFILE"], out_lib=PROF_LIB)
    moe.LIB_PATH = PROF_LIB
    L = moe.lib()
    L.moe_debug_phase_mx.argtypes = [ctypes.c_void_p]
    L.moe_debug_phase_bf.argtypes = [ctypes.c_void_p]
    dev = torch.device("cuda")
    print("| workload | precision | launch us | " + " | ".join(PHASES) + " |")
    print("|---|---|---" + "|---" * len(PHASES) + "|")
    for name in argv or ["decode", "one_token_per_expert_ep1", "one_token_per_expert_ep4"]:
        cfg = synth.config(name)
        T, H, I, E, k, e0, e1 = synth.dims_of(cfg)
        n = e1 - e0
        assert T * k <= moe.FUSED_MAX_PAIRS, name
        inp = synth.make_inputs(cfg)
        g = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)
        x, lg, wg, wu, wd = (g(inp[nm]) for nm in ("x", "logits", "w_gate", "w_up", "w_down"))
        wq = {}
        for key, w_, r_, K_ in (("g", wg, n * I, H), ("u", wu, n * I, H), ("d", wd, n * H, I)):
            q_ = torch.empty((r_, K_), dtype=torch.uint8, device=dev)
            s_ = torch.empty((r_, K_ // 32), dtype=torch.uint8, device=dev)
            moe.moe_quantize_mxfp8(w_, r_, K_, q_, s_)
            wq[key] = (q_, s_)
        out = torch.empty((T, H), dtype=torch.float32, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        wsb = moe.alloc_workspace(moe.moe_workspace_size(cfg))
        wsm = moe.alloc_workspace(moe.moe_layer_mxfp8_workspace_size(cfg))
        runs = (("bf16", lambda: moe.moe_layer(cfg, x, lg, wg, wu, wd, out, wsb, status=status), L.moe_debug_phase_bf),
                ("mxfp8", lambda: moe.moe_layer_mxfp8(cfg, x, lg, wq["g"], wq["u"], wq["d"], out, wsm, status=status),
                 L.moe_debug_phase_mx))
        for prec, launch, read in runs:
            per = [[] for _ in PHASES]
            total = []
            for rep_ in range(8):
                flush.zero_()
                torch.cuda.synchronize()
                launch()
                torch.cuda.synchronize()
                assert int(status.item()) == 0
                buf = (ctypes.c_ulonglong * (1024 * 12))()
                assert read(buf) == 0
                ts = np.frombuffer(buf, dtype=np.uint64).reshape(1024, 12)[:torch.cuda.get_device_properties(0)
                                                                          .multi_processor_count, :11].astype(np.int64)
                if rep_ < 2:
                    continue
                for i in range(len(PHASES)):
                    per[i].append((ts[:, i + 1].max() - ts[:, i].max()) / 1e3)
                total.append((ts[:, 10].max() - ts[:, 0].min()) / 1e3)
            print(f"| {name} | {prec} | {statistics.median(total):.1f} | " +
                  " | ".join(f"{statistics.median(v):.1f}" for v in per) + " |", flush=True)


def roles(argv):
    import torch

    import expert_routing_dispatch_gb300 as moe
    from expert_routing_dispatch_gb300 import _build

    _build.build(force=True, extra_flags=["-DMOE_GEMM_PROFILE"], out_lib=PROF_LIB)
    moe.LIB_PATH = PROF_LIB
    assert torch.cuda.is_available()
    names = argv or ["prefill_ep_rank", "prefill_full"]
    print("| GEMM | workload | launch ms (profile build) | tiles | MMA waits for data | MMA waits for epilogue "
          "| producer waits | epilogue waits | scale warps wait |")
    print("|---|---|---|---|---|---|---|---|---|")
    for nm in names:
        for r in measure(nm):
            sw = "—" if r[8] is None else f"{r[8]:.2f}"
            print(f"| {r[0]} | {r[1]} | {r[2]:.4f} | {r[3]} | {r[4]:.2f} | {r[5]:.2f} | {r[6]:.2f} | {r[7]:.2f} | {sw} |")


if __name__ == "__main__":
    sys.path.insert(0, ROOT)
    cmd, rest = (sys.argv[1], sys.argv[2:]) if len(sys.argv) > 1 else ("roles", [])
    {"roles": roles, "steps": steps, "phases": phases}[cmd](rest)
