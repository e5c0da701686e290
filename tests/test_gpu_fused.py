"""The fused single-launch layer (moe_layer with T*k <= MOE_FUSED_MAX_PAIRS):
bit-identical to the split entry points composed by hand, correct against the
oracle around the fused/split threshold, and its grid-barrier timeout reported
as a device status (the wait runs out; nothing faults or hangs)."""
import time

import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import OUT_TOL, bf16_h_bound, dev, host, inputs, rel_err, sample_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import torch

    import expert_routing_dispatch_gb300 as m

    assert torch.cuda.is_available()
    m.lib()
    return m


def small(T, H, I, E, k, e0, e1, seed=3):
    n = e1 - e0
    return dict(x=synth.normal_bf16(seed, synth.TID_X, (T, H), 1.0),
                logits=synth.normal_f32(seed, synth.TID_LOGITS, (T, E)),
                w_gate=synth.normal_bf16(seed, synth.TID_W_GATE, (n, I, H), 0.05, start=e0 * I * H),
                w_up=synth.normal_bf16(seed, synth.TID_W_UP, (n, I, H), 0.05, start=e0 * I * H),
                w_down=synth.normal_bf16(seed, synth.TID_W_DOWN, (n, H, I), 0.05, start=e0 * H * I))


def layer(moe, dims, inp):
    import torch

    T, H, k = dims.T, dims.H, dims.k
    out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = moe.alloc_workspace(moe.moe_workspace_size(dims))
    moe.moe_layer(dims, dev(inp["x"]), dev(inp["logits"]), dev(inp["w_gate"]), dev(inp["w_up"]),
                  dev(inp["w_down"]), out, ws, topk_idx=idx, topk_w=w, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return host(out), host(idx), host(w)


def split(moe, dims, inp):
    import torch

    T, H, I, k, n = dims.T, dims.H, dims.I, dims.k, dims.e1 - dims.e0
    P = T * k
    z = lambda shape, dt: torch.zeros(shape, dtype=dt, device="cuda")
    idx, w, st = z((T, k), torch.int32), z((T, k), torch.float32), z(1, torch.int32)
    counts, offsets, row_pair, pair_row = z(n, torch.int32), z(n + 1, torch.int32), z(P, torch.int32), z(P, torch.int32)
    x_perm, y_perm, out = z((P, H), torch.int16), z((P, H), torch.float32), z((T, H), torch.float32)
    moe.moe_route(dims, dev(inp["logits"]), idx, w, st)
    moe.moe_dispatch(dims, dev(inp["x"]), idx, counts, offsets, row_pair, pair_row, x_perm,
                     moe.alloc_workspace(moe.moe_dispatch_workspace_size(dims)))
    moe.moe_expert_ffn(dims, x_perm, offsets, dev(inp["w_gate"]), dev(inp["w_up"]), dev(inp["w_down"]), y_perm,
                       moe.alloc_workspace(moe.moe_expert_ffn_workspace_size(dims)), status=st)
    moe.moe_combine(dims, y_perm, pair_row, w, out)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return host(out), host(idx), host(w)


@pytest.mark.parametrize("name", ["decode", "tiny"])
def test_fused_equals_split_bit_for_bit(moe, name):
    cfg, inp = inputs(name)
    dims = moe.Dims.of(cfg)
    assert dims.T * dims.k <= moe.FUSED_MAX_PAIRS
    a, ia, wa = layer(moe, dims, inp)
    b, ib, wb = split(moe, dims, inp)
    assert np.array_equal(ia, ib) and np.array_equal(wa.view(np.uint32), wb.view(np.uint32))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("T,k", [(2048, 4), (2049, 4), (1024, 8), (1025, 8)])
def test_fused_split_threshold_against_oracle(moe, T, k):
    # T*k = 8192 runs fused, 8196 / 8200 run split; both checked against the oracle
    H, I, E, e0, e1 = 128, 128, 24, 4, 20
    inp = small(T, H, I, E, k, e0, e1)
    dims = moe.Dims(T, H, I, E, k, e0, e1)
    out, idx, w = layer(moe, dims, inp)
    st, ridx, rw = oracle.route(inp["logits"], k)
    assert np.array_equal(idx, ridx)
    assert (T * k <= moe.FUSED_MAX_PAIRS) == (T * k <= 8192)
    toks = sample_tokens(T, 96)
    st, ref = oracle.moe_layer_tokens(inp["logits"], inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"], k, e0, e1,
                                      tokens=toks)
    # off-workload shape: held to the elementwise bound of rounding h to bf16
    bound = bf16_h_bound(inp, k, e0, e1, toks, ridx, rw) + 1e-6 * np.abs(ref).max()
    diff = np.abs(out[toks].astype(np.float64) - ref)
    err, rms = rel_err(out[toks], ref)
    print(f"FUSED-THRESHOLD T={T} k={k} max|gpu-oracle|/RMS = {err / rms:.3e}, max err/bound = {(diff / bound).max():.3f}")
    assert np.all(diff <= bound)


def test_stalled_grid_barrier_reports_timeout_and_context_survives(moe):
    import torch

    cfg, inp = inputs("tiny")
    dims = moe.Dims.of(cfg)
    T, H = dims.T, dims.H
    out = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = moe.alloc_workspace(moe.moe_workspace_size(dims))
    t0 = time.time()
    moe.moe_testing_layer_stalled_barrier(dims, dev(inp["x"]), dev(inp["logits"]), dev(inp["w_gate"]),
                                          dev(inp["w_up"]), dev(inp["w_down"]), out, ws, status=st)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert int(st.item()) == 6  # MOE_ERR_TIMEOUT
    assert elapsed < 30
    # the context is still usable: a normal call afterwards is correct
    a, _, _ = layer(moe, dims, inp)
    st_o, ref = oracle.moe_layer_tokens(inp["logits"], inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"], dims.k,
                                        dims.e0, dims.e1)
    err, rms = rel_err(a, ref)
    assert err <= OUT_TOL * rms


@pytest.mark.parametrize("name", ["prefill_ep_rank", "skewed"])
def test_layer_split_path_equals_split_entries(moe, name):
    # moe_layer above the fused threshold runs the router with the dispatch histograms
    # and both GEMMs in one launch; composing the public entries must give the same bytes
    cfg, inp = inputs(name)
    dims = moe.Dims.of(cfg)
    assert dims.T * dims.k > moe.FUSED_MAX_PAIRS
    a, ia, wa = layer(moe, dims, inp)
    b, ib, wb = split(moe, dims, inp)
    assert np.array_equal(ia, ib) and np.array_equal(wa.view(np.uint32), wb.view(np.uint32))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("T", [256, 257])
def test_fused_top32_at_threshold(moe, T):
    # k = 32 (the largest slot count): T*k = 8192 runs fused (every CTA's slice holds up to
    # 64 pairs), 8224 runs split; both equal the split entries and the oracle
    H, I, E, k, e0, e1 = 128, 128, 40, 32, 4, 36
    inp = small(T, H, I, E, k, e0, e1, seed=9)
    dims = moe.Dims(T, H, I, E, k, e0, e1)
    assert (T * k <= moe.FUSED_MAX_PAIRS) == (T == 256)
    out, idx, w = layer(moe, dims, inp)
    ref_split, ridx_s, rw_s = split(moe, dims, inp)
    assert np.array_equal(idx, ridx_s) and np.array_equal(out.view(np.uint32), ref_split.view(np.uint32))
    st, ridx, rw = oracle.route(inp["logits"], k)
    assert np.array_equal(idx, ridx)
    toks = sample_tokens(T, 64)
    st, ref = oracle.moe_layer_tokens(inp["logits"], inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"], k, e0, e1,
                                      tokens=toks)
    bound = bf16_h_bound(inp, k, e0, e1, toks, ridx, rw) + 1e-6 * np.abs(ref).max()
    assert np.all(np.abs(out[toks].astype(np.float64) - ref) <= bound)
    if T * k <= moe.FUSED_MAX_PAIRS:  # dispatch by TMA row gather on the same shape
        import torch

        o2 = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
        stt = torch.zeros(1, dtype=torch.int32, device="cuda")
        moe.moe_layer_gather(dims, dev(inp["x"]), dev(inp["logits"]), dev(inp["w_gate"]), dev(inp["w_up"]),
                             dev(inp["w_down"]), o2, moe.alloc_workspace(moe.moe_workspace_size(dims)), status=stt)
        torch.cuda.synchronize()
        assert int(stt.item()) == 0
        assert np.array_equal(host(o2).view(np.uint32), out.view(np.uint32))
