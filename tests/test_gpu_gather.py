"""Dispatch by TMA row gather (moe_layer_gather): the fused layer with no grouped
copy of x, the gate/up GEMM loading its token rows from x by tile::gather4.  It
must be bit-identical to moe_layer (the same bytes reach the same operand tiles),
including m-tiles whose rows run past an expert's count, and it is checked
against the oracle on a shape with several m-tiles per expert."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import bf16_h_bound, dev, host, inputs, rel_err, sample_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import torch

    import expert_routing_dispatch_gb300 as m

    assert torch.cuda.is_available()
    m.lib()
    return m


def small(T, H, I, E, k, e0, e1, seed=5):
    n = e1 - e0
    return dict(x=synth.normal_bf16(seed, synth.TID_X, (T, H), 1.0),
                logits=synth.normal_f32(seed, synth.TID_LOGITS, (T, E)),
                w_gate=synth.normal_bf16(seed, synth.TID_W_GATE, (n, I, H), 0.05, start=e0 * I * H),
                w_up=synth.normal_bf16(seed, synth.TID_W_UP, (n, I, H), 0.05, start=e0 * I * H),
                w_down=synth.normal_bf16(seed, synth.TID_W_DOWN, (n, H, I), 0.05, start=e0 * H * I))


def run(moe, dims, inp, gather):
    import torch

    T, H, k = dims.T, dims.H, dims.k
    out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = moe.alloc_workspace(moe.moe_workspace_size(dims))
    ws.fill_(0xFF)  # the gathered path must not depend on the x_perm part of the workspace
    fn = moe.moe_layer_gather if gather else moe.moe_layer
    fn(dims, dev(inp["x"]), dev(inp["logits"]), dev(inp["w_gate"]), dev(inp["w_up"]), dev(inp["w_down"]), out, ws,
       topk_idx=idx, topk_w=w, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return host(out), host(idx), host(w)


@pytest.mark.parametrize("name", ["tiny", "decode", "one_token_per_expert_ep1", "one_token_per_expert_ep4"])
def test_gather_equals_copy_bit_for_bit(moe, name):
    cfg, inp = inputs(name)
    dims = moe.Dims.of(cfg)
    assert dims.T * dims.k <= moe.FUSED_MAX_PAIRS
    a, ia, wa = run(moe, dims, inp, True)
    b, ib, wb = run(moe, dims, inp, False)
    assert np.array_equal(ia, ib) and np.array_equal(wa.view(np.uint32), wb.view(np.uint32))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("T,k,E,e0,e1", [(512, 8, 24, 4, 20), (1024, 8, 9, 0, 9), (37, 3, 5, 1, 4)])
def test_gather_several_m_tiles_against_oracle(moe, T, k, E, e0, e1):
    # ~170, ~910 and ~22 rows per local expert: m-tiles of 32 rows with ragged last tiles
    H, I = 256, 192
    inp = small(T, H, I, E, k, e0, e1)
    dims = moe.Dims(T, H, I, E, k, e0, e1)
    a, ia, wa = run(moe, dims, inp, True)
    b, _, _ = run(moe, dims, inp, False)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    st, ridx, rw = oracle.route(inp["logits"], k)
    assert np.array_equal(ia, ridx)
    toks = sample_tokens(T, 64)
    st, ref = oracle.moe_layer_tokens(inp["logits"], inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"], k, e0, e1,
                                      tokens=toks)
    bound = bf16_h_bound(inp, k, e0, e1, toks, ridx, rw) + 1e-6 * np.abs(ref).max()
    diff = np.abs(a[toks].astype(np.float64) - ref)
    err, rms = rel_err(a[toks], ref)
    print(f"GATHER T={T} k={k} E={E} max|gpu-oracle|/RMS = {err / rms:.3e}, max err/bound = {(diff / bound).max():.3f}")
    assert np.all(diff <= bound)
