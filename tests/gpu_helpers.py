"""Shared helpers of the GPU parity tests: move seeded host inputs to the device,
call the C-ABI steps, and compare against the oracle.  The oracle only ever sees
host arrays made by `synth` or by `oracle` itself."""
import functools

import numpy as np

import oracle
import synth

WEIGHT_TOL = lambda k: (k + 8) * 2.0 ** -24  # |w_gpu - w_oracle|, fp32 expf/sum/div vs fp64
OUT_TOL = 2e-2  # max |gpu - oracle| <= OUT_TOL * RMS(oracle)


def dev(a, device="cuda"):
    import torch

    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device)


def host(t, dtype=None):
    a = t.detach().cpu().numpy()
    if dtype is not None:
        a = a.view(dtype)
    return a


@functools.lru_cache(maxsize=8)
def inputs(name, **over):
    cfg = synth.config(name, **dict(over))
    return cfg, synth.make_inputs(cfg)


@functools.lru_cache(maxsize=8)
def oracle_routing(name, **over):
    cfg, inp = inputs(name, **over)
    st, idx, w = oracle.route(inp["logits"], cfg["k"])
    assert st == 0
    d = oracle.dispatch(idx, cfg["e0"], cfg["e1"])
    return idx, w, d


def sample_tokens(T, n, seed=0):
    """All tokens when T <= n, else the first, the last and n-2 seeded others."""
    if T <= n:
        return np.arange(T, dtype=np.int64)
    rest = synth.uniform_int(seed, synth.TID_AUX + 7, n - 2, T)
    return np.unique(np.concatenate([[0, T - 1], rest]).astype(np.int64))


def sample_rows(offsets, n_per_expert=3, extra=64, seed=0):
    """First and last row of every non-empty expert plus seeded extra rows."""
    off = np.asarray(offsets)
    R = int(off[-1])
    rows = []
    for e in range(off.size - 1):
        if off[e + 1] > off[e]:
            rows += [off[e], off[e + 1] - 1]
            if n_per_expert > 2 and off[e + 1] - off[e] > 2:
                rows.append((off[e] + off[e + 1]) // 2)
    if R > 0:
        rows += list(synth.uniform_int(seed, synth.TID_AUX + 8, extra, R))
    return np.unique(np.asarray(rows, dtype=np.int64))


def parity_rows(offsets, at_least=2048, seed=0):
    """Grouped rows for a parity check: every row when R <= at_least; else the
    first, middle and last row of every non-empty expert plus seeded rows, at
    least `at_least` distinct rows in all."""
    off = np.asarray(offsets, np.int64)
    R = int(off[-1])
    if R <= at_least:
        return np.arange(R, dtype=np.int64)
    rows = set()
    for e in range(off.size - 1):
        if off[e + 1] > off[e]:
            rows.update((int(off[e]), int((off[e] + off[e + 1]) // 2), int(off[e + 1] - 1)))
    draw = 0
    while len(rows) < at_least:
        rows.update(int(r) for r in synth.uniform_int(seed + draw, synth.TID_AUX + 8, at_least, R))
        draw += 1
    return np.asarray(sorted(rows), dtype=np.int64)


def parity_tokens(T, at_least=2048, seed=0):
    """Every token when T <= at_least, else the first, the last and seeded others,
    at least `at_least` distinct tokens in all."""
    if T <= at_least:
        return np.arange(T, dtype=np.int64)
    toks = {0, T - 1}
    draw = 0
    while len(toks) < at_least:
        toks.update(int(t) for t in synth.uniform_int(seed + draw, synth.TID_AUX + 7, at_least, T))
        draw += 1
    return np.asarray(sorted(toks), dtype=np.int64)


def bf16_h_bound(inp, k, e0, e1, tokens, idx, w):
    """Elementwise bound of |gpu - oracle| implied by the GPU's arithmetic: h is
    rounded to bf16 (unit roundoff u = 2^-8) before the down GEMM, everything
    else is fp32 (relative errors ~2^-20 here, below 10% of the main term), so
    |err[t]| <= 1.1 * u * sum_j w_tj * (|W_down[e_j]| @ |h_tj|)."""
    bf = synth.bf16_to_f32
    H = inp["x"].shape[1]
    out = np.zeros((len(tokens), H))
    for q, t in enumerate(tokens):
        xt = bf(inp["x"][t]).astype(np.float64)
        for j in range(k):
            e = int(idx[t, j])
            if not (e0 <= e < e1):
                continue
            g = bf(inp["w_gate"][e - e0]).astype(np.float64) @ xt
            u = bf(inp["w_up"][e - e0]).astype(np.float64) @ xt
            h = np.abs(g / (1.0 + np.exp(-g)) * u)
            out[q] += float(w[t, j]) * (np.abs(bf(inp["w_down"][e - e0]).astype(np.float64)) @ h)
    return 1.1 * 2.0 ** -8 * out


def rel_err(got, ref):
    rms = float(np.sqrt(np.mean(np.asarray(ref, np.float64) ** 2)))
    err = float(np.abs(np.asarray(got, np.float64) - ref).max()) if np.size(ref) else 0.0
    return err, rms


# ---------------------------------------------------------------- MXFP8 rounding ambiguity
_E4M3 = []


def e4m3_magnitudes():
    """The non-negative finite E4M3 values in code order (codes 0..126, ascending),
    read from the oracle's dequantiser at block scale 2^0."""
    if not _E4M3:
        q = np.zeros((1, 128), np.uint8)
        q[0, :127] = np.arange(127)
        s = np.full((1, 4), 127, np.uint8)
        _E4M3.append(oracle.mxfp8_dequantize(q, s)[0, :127])
    return _E4M3[0]


def mx_ambiguity(h64, hs, rel_tau=2.0 ** -10, abs_tau=2.0 ** -16, scale_tau=2.0 ** -14):
    """Which E4M3 codes of the MXFP8 quantisation of h64 (fp64 [rows, I]; the
    oracle's block scale codes hs [rows, I/32]) a kernel that computes h in fp32,
    with another summation order, may legitimately round the other way.

    An element is ambiguous when its scaled value v = |h| / X lies within
    max(rel_tau * step, abs_tau * block max) of the rounding midpoint between its
    two neighbouring E4M3 values (step = their spacing): there the fp32 value can
    fall on either side.  A block is scale-ambiguous when its largest |h| lies
    within a relative scale_tau of a power of two (the UE8M0 scale can then differ
    by one), and all its elements count as ambiguous.  Returns (amb [rows, I],
    delta [rows, I]: the most an ambiguous element's dequantised value can differ
    from the oracle's, scale_amb [rows, I/32])."""
    grid = e4m3_magnitudes()
    rows, I = h64.shape
    X = 2.0 ** (np.repeat(hs.astype(np.float64), 32, axis=1) - 127)
    v = np.abs(h64) / X
    j = np.clip(np.searchsorted(grid, v, side="left"), 1, grid.size - 1)
    a, b = grid[j - 1], grid[j]
    step = b - a
    dist = np.abs(v - 0.5 * (a + b))
    vmax = np.repeat(v.reshape(rows, I // 32, 32).max(axis=2), 32, axis=1)
    amb = dist <= np.maximum(rel_tau * step, abs_tau * vmax)
    delta = step * X
    amax = np.abs(h64).reshape(rows, I // 32, 32).max(axis=2)
    with np.errstate(divide="ignore"):
        lg = np.log2(np.where(amax > 0, amax, 1.0))
    scale_amb = (amax > 0) & (np.abs(lg - np.round(lg)) * np.log(2.0) <= scale_tau)
    if scale_amb.any():
        sa = np.repeat(scale_amb, 32, axis=1)
        # at half the scale the values double and the largest saturate at 448
        extra = 2.0 * step * X + np.maximum(0.0, 2.0 * v - 448.0) * X / 2.0
        amb = amb | sa
        delta = np.where(sa, np.maximum(delta, extra), delta)
    return amb, np.where(amb, delta, 0.0), scale_amb


def mx_down_bound(rows, offsets, wd, dh):
    """Elementwise bound on how far the down GEMM's output rows move when their h
    rows move by at most dh (fp64 [len(rows), I]): |W_down[e]| |dh| per row, with
    W_down the dequantised MXFP8 weights (q, s) of each row's expert."""
    q, s = wd
    e_of = np.searchsorted(np.asarray(offsets), rows, side="right") - 1
    out = np.zeros((len(rows), q.shape[1]))
    for e in np.unique(e_of):
        sel = np.nonzero(e_of == e)[0]
        if not dh[sel].any():
            continue
        out[sel] = dh[sel] @ np.abs(oracle.mxfp8_dequantize(q[e], s[e])).T
    return out
