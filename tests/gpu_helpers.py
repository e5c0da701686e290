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
