"""Pins of the oracle's expert FFN and combine steps (CPU only): a textbook
SwiGLU MLP written independently in numpy, closed forms with identity-like
weights, routing-independence with identical experts, the dense masked
formula, and the range-decomposition invariant (the outputs of disjoint local
ranges sum to the full-range output)."""
import math

import numpy as np
import pytest

import oracle
import synth

bf = synth.bf16_to_f32


def textbook_swiglu(x, wg, wu, wd):
    """Dense SwiGLU MLP in fp64: W_d (silu(W_g x) * (W_u x)); silu written via tanh."""
    g = wg @ x
    u = wu @ x
    silu = 0.5 * g * (1.0 + np.tanh(0.5 * g))
    return wd @ (silu * u)


def small_problem(T, H, I, E, k, seed, w_std=0.1):
    x = synth.normal_bf16(seed, synth.TID_AUX + 1, (T, H), 1.0)
    lg = synth.normal_f32(seed, synth.TID_AUX + 2, (T, E))
    wg = synth.normal_bf16(seed, synth.TID_AUX + 3, (E, I, H), w_std)
    wu = synth.normal_bf16(seed, synth.TID_AUX + 4, (E, I, H), w_std)
    wd = synth.normal_bf16(seed, synth.TID_AUX + 5, (E, H, I), w_std)
    return x, lg, wg, wu, wd


def dense_masked_reference(x, lg, wg, wu, wd, k, e0, e1):
    """out_t = sum_e [e picked and e in range] * w_te * FFN_e(x_t), weights from the
    renormalised full softmax, selection from a full stable sort."""
    T, E = lg.shape
    out = np.zeros((T, x.shape[1]))
    xs = bf(x).astype(np.float64)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(lg[t, e]), e))[:k]
        p = np.exp(lg[t].astype(np.float64))
        p /= p.sum()
        wsel = p[order] / p[order].sum()
        for w, e in zip(wsel, order):
            if e0 <= e < e1:
                out[t] += w * textbook_swiglu(xs[t], bf(wg[e - e0]).astype(np.float64),
                                              bf(wu[e - e0]).astype(np.float64),
                                              bf(wd[e - e0]).astype(np.float64))
    return out


def test_single_expert_is_textbook_mlp():
    T, H, I = 12, 32, 24
    x, lg, wg, wu, wd = small_problem(T, H, I, 1, 1, seed=1)
    st, out = oracle.moe_layer_tokens(lg, x, wg, wu, wd, 1, 0, 1)
    assert st == 0
    ref = np.stack([textbook_swiglu(bf(x[t]).astype(np.float64), bf(wg[0]).astype(np.float64),
                                    bf(wu[0]).astype(np.float64), bf(wd[0]).astype(np.float64))
                    for t in range(T)])
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_identity_weights_closed_form():
    # I = H, W_gate = c*Id, W_up = W_down = Id  =>  out = x * silu(c x)
    H, c = 16, 0.5
    T = 20
    eye = synth.f32_to_bf16(np.eye(H, dtype=np.float32))
    wg = synth.f32_to_bf16(c * np.eye(H, dtype=np.float32))[None]
    x = synth.normal_bf16(3, synth.TID_AUX, (T, H), 2.0)
    lg = np.zeros((T, 1), np.float32)
    st, out = oracle.moe_layer_tokens(lg, x, wg, eye[None], eye[None], 1, 0, 1)
    assert st == 0
    xf = bf(x).astype(np.float64)
    for t in range(T):
        for h in range(H):
            z = c * xf[t, h]
            assert abs(out[t, h] - xf[t, h] * z / (1.0 + math.exp(-z))) <= 1e-14 * (1 + abs(out[t, h]))


def test_identical_experts_independent_of_routing():
    T, H, I, E, k = 16, 32, 16, 6, 3
    x, lg, wg, wu, wd = small_problem(T, H, I, 1, 1, seed=2)
    rep = lambda w: np.repeat(w, E, axis=0)
    st, out = oracle.moe_layer_tokens(synth.normal_f32(9, synth.TID_AUX, (T, E)), x,
                                      rep(wg), rep(wu), rep(wd), k, 0, E)
    assert st == 0
    st1, ref = oracle.moe_layer_tokens(lg[:, :1], x, wg, wu, wd, 1, 0, 1)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


@pytest.mark.parametrize("e0,e1", [(0, 6), (2, 5), (5, 6)])
def test_dense_masked_formula(e0, e1):
    T, H, I, E, k = 10, 24, 16, 6, 3
    x, lg, wg, wu, wd = small_problem(T, H, I, E, k, seed=4)
    st, out = oracle.moe_layer_tokens(lg, x, wg[e0:e1], wu[e0:e1], wd[e0:e1], k, e0, e1)
    assert st == 0
    ref = dense_masked_reference(x, lg, wg[e0:e1], wu[e0:e1], wd[e0:e1], k, e0, e1)
    assert np.allclose(out, ref, rtol=1e-11, atol=1e-12 * max(np.abs(ref).max(), 1e-30))


def test_range_decomposition():
    T, H, I, E, k = 40, 32, 16, 8, 3
    x, lg, wg, wu, wd = small_problem(T, H, I, E, k, seed=5)
    st, full = oracle.moe_layer_tokens(lg, x, wg, wu, wd, k, 0, E)
    acc = np.zeros_like(full)
    for e0 in range(0, E, 2):
        st, part = oracle.moe_layer_tokens(lg, x, wg[e0:e0 + 2], wu[e0:e0 + 2], wd[e0:e0 + 2], k, e0, e0 + 2)
        assert st == 0
        acc += part
    rms = np.sqrt((full ** 2).mean())
    assert np.abs(acc - full).max() <= 1e-12 * rms


def test_grouped_rows_match_textbook():
    T, H, I, E, k = 30, 32, 16, 4, 2
    x, lg, wg, wu, wd = small_problem(T, H, I, E, k, seed=6)
    st, idx, w = oracle.route(lg, k)
    d = oracle.dispatch(idx, 1, 4)
    xp = x[d["row_pair"] // k]
    y = oracle.expert_ffn_rows(xp, d["offsets"], wg[1:4], wu[1:4], wd[1:4])
    for r in range(d["R"]):
        e = int(np.searchsorted(d["offsets"], r, side="right") - 1)
        ref = textbook_swiglu(bf(xp[r]).astype(np.float64), bf(wg[1 + e]).astype(np.float64),
                              bf(wu[1 + e]).astype(np.float64), bf(wd[1 + e]).astype(np.float64))
        assert np.allclose(y[r], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    # rows past R are zero
    y2 = oracle.expert_ffn_rows(xp, d["offsets"], wg[1:4], wu[1:4], wd[1:4], 0, d["R"] + 3)
    assert (y2[d["R"]:] == 0).all()


def test_combine_is_slot_ordered_weighted_gather():
    T, H, k, E = 25, 16, 3, 8
    lg = synth.normal_f32(8, synth.TID_AUX, (T, E))
    st, idx, w64 = oracle.route(lg, k)
    d = oracle.dispatch(idx, 2, 7)
    yp = synth.normal_f32(8, synth.TID_AUX + 1, (max(d["R"], 1), H))
    w32 = w64.astype(np.float32)
    out = oracle.combine_tokens(yp, d["pair_row"], w32)
    yf = yp.astype(np.float64)
    for t in range(T):
        ref = np.zeros(H)
        for j in range(k):
            r = d["pair_row"][t * k + j]
            if r >= 0:
                ref = ref + float(w32[t, j]) * yf[r]
        assert np.array_equal(out[t], ref) or np.allclose(out[t], ref, rtol=1e-15, atol=0)
    no_local = [t for t in range(T) if (d["pair_row"][t * k:(t + 1) * k] < 0).all()]
    assert all((out[t] == 0).all() for t in no_local)


def test_layer_nonfinite_status():
    T, H, I, E, k = 4, 16, 16, 4, 2
    x, lg, wg, wu, wd = small_problem(T, H, I, E, k, seed=9)
    lg = lg.copy()
    lg[1, 2] = np.nan
    st, _ = oracle.moe_layer_tokens(lg, x, wg, wu, wd, k, 0, E)
    assert st == oracle.NONFINITE


def test_rowlist_equals_row_range():
    T, H, I, E, k = 20, 32, 16, 3, 2
    x, lg, wg, wu, wd = small_problem(T, H, I, E, k, seed=10)
    st, idx, w = oracle.route(lg, k)
    d = oracle.dispatch(idx, 0, 3)
    xp = x[d["row_pair"] // k]
    full = oracle.expert_ffn_rows(xp, d["offsets"], wg, wu, wd)
    rows = np.array([0, 5, d["R"] - 1, 3], np.int64)
    assert np.array_equal(oracle.expert_ffn_rowlist(xp, d["offsets"], wg, wu, wd, rows), full[rows])
