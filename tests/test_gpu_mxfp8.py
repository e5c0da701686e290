"""GPU parity of the MXFP8 expert path ("MoE GEMM" section of "Hosting Qwen on
Blackwell": the deployed expert GEMMs run in MXFP8, read as OCP MX v1.0 MXFP8)
against the oracle, through the C ABI.

Bars:
- quantisation (moe_quantize_mxfp8) is bit-exact: E4M3 codes and UE8M0 scales;
- h (quantised to MXFP8 in the gate/up epilogue from fp32 values): the E4M3 code
  and the UE8M0 scale are integers that floating point decides, and the kernel
  decides them from an fp32 h summed in another order than the oracle's fp64 h.
  So the codes and scales must equal the oracle's except where the oracle's h
  lies within a small band of a rounding midpoint (or its block maximum within a
  small band of a power of two), where either neighbour is a correct rounding
  (gpu_helpers.mx_ambiguity); there the dequantised values may differ by at most
  that spacing;
- the down GEMM alone (the oracle fed the GPU's own quantised h): within 1e-3 *
  RMS, i.e. fp32 accumulation (a wrong scale anywhere would be a factor of 2);
- the expert FFN rows and the layer output against the oracle's own MXFP8
  pipeline: elementwise within |W_down| applied to the largest change the
  ambiguous codes allow (zero where no code is ambiguous), plus 1e-4 * RMS for
  the fp32 arithmetic; routing bit-exact.  max |gpu - oracle| / RMS is printed.
The FFN is checked on at least 2048 grouped rows per workload (all rows when there
are fewer, always the first, middle and last row of every expert), the layer on at
least 2048 tokens (all of them when there are fewer).
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import (dev, host, inputs, mx_ambiguity, mx_down_bound, oracle_routing, parity_rows,
                         parity_tokens, rel_err)

pytestmark = pytest.mark.gpu

CONFIGS = ["tiny", "decode", "prefill_ep_rank", "skewed_rank0"]


@pytest.fixture(scope="module")
def moe():
    import torch

    import expert_routing_dispatch_gb300 as m

    assert torch.cuda.is_available()
    m.lib()
    return m


_wcache = {}


def mx_weights(name):
    """oracle MXFP8 of the config's weights: (q, s) per matrix, shaped like the bf16 weights"""
    if name not in _wcache:
        cfg, inp = inputs(name)
        out = {}
        for key in ("w_gate", "w_up", "w_down"):
            w = inp[key]
            q, s = oracle.mxfp8_quantize(w.reshape(-1, w.shape[-1]))
            out[key] = (q.reshape(w.shape), s.reshape(w.shape[:-1] + (w.shape[-1] // 32,)))
        _wcache[name] = out
    return _wcache[name]


FP32_SLACK = 1e-4  # of RMS: the fp32 accumulation of the down GEMM (measured ~3e-6)


def mx_rows_reference(xq, xs, offsets, w, rows):
    """The oracle's MXFP8 FFN of grouped rows, its h (fp64, codes, scales) and the
    ambiguity of its h codes: (y_own, h64, hq_o, hs_o, amb, delta, scale_amb,
    bound), bound = |W_down| applied to the ambiguous codes' largest change."""
    y_own, h64, hq_o, hs_o = oracle.expert_ffn_mxfp8_rowlist(xq, xs, offsets, w["w_gate"], w["w_up"], w["w_down"],
                                                             rows, want_h=True)
    amb, delta, scale_amb = mx_ambiguity(h64, hs_o)
    bound = mx_down_bound(rows, offsets, w["w_down"], delta)
    return y_own, h64, hq_o, hs_o, amb, delta, scale_amb, bound


@pytest.mark.parametrize("name", ["tiny", "prefill_ep_rank"])
def test_quantize_bit_exact(moe, name):
    import torch

    cfg, inp = inputs(name)
    for key in ("x", "w_down"):
        a = inp[key].reshape(-1, inp[key].shape[-1])[:4096]
        rows, K = a.shape
        q = torch.empty((rows, K), dtype=torch.uint8, device="cuda")
        s = torch.empty((rows, K // 32), dtype=torch.uint8, device="cuda")
        moe.moe_quantize_mxfp8(dev(a), rows, K, q, s)
        torch.cuda.synchronize()
        rq, rs = oracle.mxfp8_quantize(a)
        assert np.array_equal(host(q), rq) and np.array_equal(host(s), rs), key


def test_quantize_special_values(moe):
    import torch

    # zero block, ties, saturation, signed zero, subnormal codes, a block near the bottom of the scale range
    vals = np.zeros((4, 32), np.float32)
    vals[1, :6] = [256.0, 17.0, 19.0, -17.0, -(2.0 ** -100), 500.0]
    vals[2] = np.linspace(-1.0, 1.0, 32) * 2.0 ** -8
    vals[2, 0] = 448.0 * 2.0 ** -8
    vals[3] = np.linspace(0, 1, 32) * 2.0 ** -118
    a = synth.f32_to_bf16(vals)
    q = torch.empty((4, 32), dtype=torch.uint8, device="cuda")
    s = torch.empty((4, 1), dtype=torch.uint8, device="cuda")
    moe.moe_quantize_mxfp8(dev(a), 4, 32, q, s)
    torch.cuda.synchronize()
    rq, rs = oracle.mxfp8_quantize(a)
    assert np.array_equal(host(q), rq) and np.array_equal(host(s), rs)


def run_ffn(moe, name):
    import torch

    cfg, inp = inputs(name)
    T, H, I, E, k, e0, e1 = synth.dims_of(cfg)
    _, _, d = oracle_routing(name)
    P, R = T * k, d["R"]
    xq_t, xs_t = oracle.mxfp8_quantize(inp["x"])
    xq = np.zeros((P, H), np.uint8)
    xs = np.zeros((P, H // 32), np.uint8)
    xq[:R] = xq_t[d["row_pair"] // k]
    xs[:R] = xs_t[d["row_pair"] // k]
    w = mx_weights(name)
    dw = {key: (dev(q), dev(s)) for key, (q, s) in w.items()}
    y = torch.full((P, H), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = moe.alloc_workspace(moe.moe_expert_ffn_mxfp8_workspace_size(cfg))
    moe.moe_expert_ffn_mxfp8(cfg, dev(xq), dev(xs), dev(d["offsets"]), dw["w_gate"], dw["w_up"], dw["w_down"], y, ws,
                             status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    hq_off = (P * I + 255) // 256 * 256
    wsh = host(ws)
    hq = wsh[:P * I].reshape(P, I)
    hs = wsh[hq_off:hq_off + P * (I // 32)].reshape(P, I // 32)
    return cfg, d, xq, xs, w, host(y), hq, hs


@pytest.mark.parametrize("name", CONFIGS)
def test_mx_expert_ffn(moe, name):
    cfg, d, xq, xs, w, y, hq, hs = run_ffn(moe, name)
    R = d["R"]
    rows = parity_rows(d["offsets"], at_least=2048)
    if rows.size == 0:
        return
    y_own, h64, hq_o, hs_o, amb, delta, scale_amb, bound = mx_rows_reference(xq, xs, d["offsets"], w, rows)
    # h codes and scales: equal to the oracle's except where either rounding is correct
    assert ((hs[rows] == hs_o) | scale_amb).all()
    assert ((hq[rows] == hq_o) | amb).all(), int(((hq[rows] != hq_o) & ~amb).sum())
    hg, ho = oracle.mxfp8_dequantize(hq[rows], hs[rows]), oracle.mxfp8_dequantize(hq_o, hs_o)
    assert (np.abs(hg - ho) <= delta * (1 + 1e-12)).all()
    flips = float(np.mean(hq[rows] != hq_o))
    # the down GEMM alone (fed the GPU's own h codes)
    y_gpu_h = oracle.expert_ffn_mxfp8_rowlist(xq, xs, d["offsets"], w["w_gate"], w["w_up"], w["w_down"], rows,
                                              h_in=(hq[rows], hs[rows]))
    e_down, rms_down = rel_err(y[rows], y_gpu_h)
    # the whole FFN against the oracle's own MXFP8 pipeline
    e_all, rms_all = rel_err(y[rows], y_own)
    diff = np.abs(y[rows].astype(np.float64) - y_own)
    print(f"PARITY mxfp8 ffn {cfg['name']} rows {rows.size} of {R}: h codes ambiguous {amb.mean():.4%}, flipped "
          f"{flips:.4%}; down-only max/RMS {e_down / rms_down:.2e}; ffn max/RMS {e_all / rms_all:.2e}, "
          f"max err/(bound + slack) {(diff / (bound + FP32_SLACK * rms_all)).max():.3f}")
    assert e_down <= 1e-3 * rms_down
    assert (diff <= bound + FP32_SLACK * rms_all).all()


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill_ep_rank", "skewed"])
def test_mx_layer(moe, name):
    import torch

    cfg, inp = inputs(name)
    T, H, I, E, k, e0, e1 = synth.dims_of(cfg)
    idx_o, w_o, d = oracle_routing(name)
    w = mx_weights(name)
    dw = {key: (dev(q), dev(s)) for key, (q, s) in w.items()}
    out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    wt = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = moe.alloc_workspace(moe.moe_layer_mxfp8_workspace_size(cfg))
    moe.moe_layer_mxfp8(cfg, dev(inp["x"]), dev(inp["logits"]), dw["w_gate"], dw["w_up"], dw["w_down"], out, ws,
                        topk_idx=idx, topk_w=wt, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(host(idx), idx_o)
    toks = parity_tokens(T, 2048)
    # oracle: MXFP8 FFN of every local slot of the sampled tokens, combined in slot order
    xq_t, xs_t = oracle.mxfp8_quantize(inp["x"])
    P = T * k
    pr = d["pair_row"]
    rows = np.unique(np.array([pr[t * k + j] for t in toks for j in range(k) if pr[t * k + j] >= 0], np.int64))
    got = host(out)[toks]
    if rows.size == 0:
        assert (got == 0).all()
        return
    xq = np.zeros((P, H), np.uint8)
    xs = np.zeros((P, H // 32), np.uint8)
    xq[:d["R"]] = xq_t[d["row_pair"] // k]
    xs[:d["R"]] = xs_t[d["row_pair"] // k]
    y_rows, _, _, _, amb, _, _, bound_rows = mx_rows_reference(xq, xs, d["offsets"], w, rows)
    y_perm = np.zeros((P, H), np.float32)
    y_perm[rows] = y_rows.astype(np.float32)
    ref = oracle.combine_tokens(y_perm, pr, w_o.astype(np.float32), tokens=toks)
    b_perm = np.zeros((P, H), np.float32)
    b_perm[rows] = bound_rows.astype(np.float32)
    bound = oracle.combine_tokens(b_perm, pr, np.abs(w_o).astype(np.float32), tokens=toks)
    err, rms = rel_err(got, ref)
    diff = np.abs(got.astype(np.float64) - ref)
    # context only: the bf16 oracle of the same tokens
    st, ref16 = oracle.moe_layer_tokens(inp["logits"], inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"], k, e0, e1,
                                        tokens=toks)
    e16, rms16 = rel_err(got, ref16)
    print(f"PARITY mxfp8 layer {name} tokens {toks.size} of {T}: max|gpu-oracle_mx|/RMS = {err / rms:.3e}, max "
          f"err/(bound + slack) {(diff / (bound + FP32_SLACK * rms)).max():.3f} (vs the bf16 oracle: {e16 / rms16:.3e})")
    assert (diff <= bound * (1 + 1e-6) + FP32_SLACK * rms).all()


@pytest.mark.parametrize("dims", [
    (1, 128, 128, 4, 1, 0, 4),        # T = 1, k = 1
    (300, 384, 640, 8, 2, 1, 5),      # I = 6.67 gate/up tiles of 96 columns, H = 2 down tiles of 192
    (513, 256, 128, 3, 1, 1, 2),      # one local expert, m-tile tail, I smaller than a gate/up tile
    (37, 128, 256, 8, 8, 2, 5),       # k = E, partial range
    (256, 128, 128, 40, 32, 4, 36),   # k = 32 at T*k = 8192: the fused launch, 64 pairs per CTA slice
])
def test_mx_layer_small_shapes(moe, dims):
    import torch

    T, H, I, E, k, e0, e1 = dims
    n = e1 - e0
    x = synth.normal_bf16(0, synth.TID_X, (T, H), 1.0)
    lg = synth.normal_f32(0, synth.TID_LOGITS, (T, E))
    wb = {key: synth.normal_bf16(0, tid, shape, 0.05, start=e0 * shape[1] * shape[2])
          for key, tid, shape in (("w_gate", synth.TID_W_GATE, (n, I, H)), ("w_up", synth.TID_W_UP, (n, I, H)),
                                  ("w_down", synth.TID_W_DOWN, (n, H, I)))}
    w = {}
    for key, a in wb.items():
        q, s = oracle.mxfp8_quantize(a.reshape(-1, a.shape[-1]))
        w[key] = (q.reshape(a.shape), s.reshape(a.shape[:-1] + (a.shape[-1] // 32,)))
    dw = {key: (dev(q), dev(s)) for key, (q, s) in w.items()}
    dims_ = moe.Dims(*dims)
    out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    wt = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = moe.alloc_workspace(moe.moe_layer_mxfp8_workspace_size(dims_))
    moe.moe_layer_mxfp8(dims_, dev(x), dev(lg), dw["w_gate"], dw["w_up"], dw["w_down"], out, ws, topk_idx=idx,
                        topk_w=wt, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    st, ridx, rw = oracle.route(lg, k)
    assert np.array_equal(host(idx), ridx)
    d = oracle.dispatch(ridx, e0, e1)
    P, R = T * k, d["R"]
    xq_t, xs_t = oracle.mxfp8_quantize(x)
    xq = np.zeros((P, H), np.uint8)
    xs = np.zeros((P, H // 32), np.uint8)
    xq[:R] = xq_t[d["row_pair"] // k]
    xs[:R] = xs_t[d["row_pair"] // k]
    y_perm = np.zeros((P, H), np.float32)
    b_perm = np.zeros((P, H), np.float32)
    if R:
        rows = np.arange(R, dtype=np.int64)
        y_rows, _, _, _, _, _, _, bound_rows = mx_rows_reference(xq, xs, d["offsets"], w, rows)
        y_perm[:R] = y_rows.astype(np.float32)
        b_perm[:R] = bound_rows.astype(np.float32)
    ref = oracle.combine_tokens(y_perm, d["pair_row"], rw.astype(np.float32))
    bound = oracle.combine_tokens(b_perm, d["pair_row"], np.abs(rw).astype(np.float32))
    got = host(out)
    if R == 0:
        assert (got == 0).all()
        return
    err, rms = rel_err(got, ref)
    diff = np.abs(got.astype(np.float64) - ref)
    print(f"PARITY mxfp8 small {dims} max|gpu-oracle_mx|/RMS = {err / rms:.3e}, max err/(bound + slack) "
          f"{(diff / (bound + FP32_SLACK * rms)).max():.3f}")
    assert (diff <= bound * (1 + 1e-6) + FP32_SLACK * rms).all()



def _mx_layer(moe, dims, inp, w):
    import torch

    T, H, I, E, k, e0, e1 = (dims.T, dims.H, dims.I, dims.E, dims.k, dims.e0, dims.e1)
    dw = {key: (dev(q), dev(s)) for key, (q, s) in w.items()}
    out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    wt = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = moe.alloc_workspace(moe.moe_layer_mxfp8_workspace_size(dims))
    moe.moe_layer_mxfp8(dims, dev(inp["x"]), dev(inp["logits"]), dw["w_gate"], dw["w_up"], dw["w_down"], out, ws,
                        topk_idx=idx, topk_w=wt, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return host(out), host(idx), host(wt)


def _mx_split_entries(moe, dims, inp, w):
    """moe_route, moe_dispatch (bf16 rows), moe_quantize_mxfp8 of the grouped rows,
    moe_expert_ffn_mxfp8 and moe_combine, composed by hand."""
    import torch

    T, H, I, E, k, e0, e1 = (dims.T, dims.H, dims.I, dims.E, dims.k, dims.e0, dims.e1)
    n, P = e1 - e0, T * k
    z = lambda shape, dt: torch.zeros(shape, dtype=dt, device="cuda")
    dw = {key: (dev(q), dev(s)) for key, (q, s) in w.items()}
    idx, wt, st = z((T, k), torch.int32), z((T, k), torch.float32), z(1, torch.int32)
    counts, offsets, row_pair, pair_row = z(n, torch.int32), z(n + 1, torch.int32), z(P, torch.int32), z(P, torch.int32)
    x_perm, y, out = z((P, H), torch.int16), z((P, H), torch.float32), z((T, H), torch.float32)
    xq, xs = z((P, H), torch.uint8), z((P, H // 32), torch.uint8)
    moe.moe_route(dims, dev(inp["logits"]), idx, wt, st)
    moe.moe_dispatch(dims, dev(inp["x"]), idx, counts, offsets, row_pair, pair_row, x_perm,
                     moe.alloc_workspace(moe.moe_dispatch_workspace_size(dims)))
    moe.moe_quantize_mxfp8(x_perm, P, H, xq, xs)
    moe.moe_expert_ffn_mxfp8(dims, xq, xs, offsets, dw["w_gate"], dw["w_up"], dw["w_down"], y,
                             moe.alloc_workspace(moe.moe_expert_ffn_mxfp8_workspace_size(dims)), status=st)
    moe.moe_combine(dims, y, pair_row, wt, out)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return host(out), host(idx), host(wt)


@pytest.mark.parametrize("name", ["decode", "tiny"])
def test_mx_fused_equals_split_bit_for_bit(moe, name):
    # T*k <= MOE_FUSED_MAX_PAIRS: moe_layer_mxfp8 is one cooperative launch (x quantised per
    # token inside it); the split entries must give the same bytes
    cfg, inp = inputs(name)
    dims = moe.Dims.of(cfg)
    assert dims.T * dims.k <= moe.FUSED_MAX_PAIRS
    w = mx_weights(name)
    a, ia, wa = _mx_layer(moe, dims, inp, w)
    b, ib, wb = _mx_split_entries(moe, dims, inp, w)
    assert np.array_equal(ia, ib) and np.array_equal(wa.view(np.uint32), wb.view(np.uint32))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_mx_layer_split_path_equals_split_entries(moe):
    # above the threshold moe_layer_mxfp8 runs its split kernels (x quantised before the row
    # copy); composing the public entries must give the same bytes
    cfg, inp = inputs("prefill_ep_rank")
    dims = moe.Dims.of(cfg)
    assert dims.T * dims.k > moe.FUSED_MAX_PAIRS
    w = mx_weights("prefill_ep_rank")
    a, ia, wa = _mx_layer(moe, dims, inp, w)
    b, ib, wb = _mx_split_entries(moe, dims, inp, w)
    assert np.array_equal(ia, ib)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
