"""Failure detection of the split grouped GEMMs without a GPU fault: the testing
entries make the first ring stage of every CTA wait for one arrival more than is
ever made, so the MMA warp's bounded mbarrier wait runs out (~1 s of clock
cycles).  Each kernel must report MOE_ERR_TIMEOUT in the status word, stop its
roles, wait for its own copies in flight, free its tensor memory and return; the
next normal call on the same context must then match the oracle."""
import time

import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import OUT_TOL, dev, host, inputs, oracle_routing, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import torch

    import expert_routing_dispatch_gb300 as m

    assert torch.cuda.is_available()
    m.lib()
    return m


def grouped_x(name):
    cfg, inp = inputs(name)
    T, H, I, E, k, e0, e1 = synth.dims_of(cfg)
    _, _, d = oracle_routing(name)
    x_perm = np.zeros((T * k, H), np.uint16)
    x_perm[:d["R"]] = inp["x"][d["row_pair"] // k]
    return cfg, inp, d, x_perm


def test_gate_up_wait_timeout_reports_status_and_context_survives(moe):
    import torch

    cfg, inp, d, x_perm = grouped_x("tiny")
    T, H, I, E, k, e0, e1 = synth.dims_of(cfg)
    P, R = T * k, d["R"]
    xp, off = dev(x_perm), dev(d["offsets"])
    wg, wu, wd = dev(inp["w_gate"]), dev(inp["w_up"]), dev(inp["w_down"])
    h = torch.zeros((P, 2 * I), dtype=torch.int16, device="cuda")  # h as bf16 hi and lo terms
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.time()
    moe.moe_testing_expert_gate_up_stalled(cfg, xp, off, wg, wu, h, status=st)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    print(f"TIMEOUT gate/up: status {int(st.item())} after {elapsed:.2f} s")
    assert int(st.item()) == 6  # MOE_ERR_TIMEOUT
    assert elapsed < 30
    # the context is still usable: a normal gate/up + down afterwards matches the oracle
    st.zero_()
    y = torch.full((P, H), float("nan"), dtype=torch.float32, device="cuda")
    moe.moe_expert_gate_up(cfg, xp, off, wg, wu, h, status=st)
    moe.moe_expert_down(cfg, h, off, wd, y, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows = np.arange(R, dtype=np.int64)
    ref = oracle.expert_ffn_rowlist(x_perm, d["offsets"], inp["w_gate"], inp["w_up"], inp["w_down"], rows)
    err, rms = rel_err(host(y)[:R], ref)
    assert err <= OUT_TOL * rms


def test_mxfp8_ffn_wait_timeout_reports_status_and_context_survives(moe):
    import torch

    cfg, inp, d, _ = grouped_x("tiny")
    T, H, I, E, k, e0, e1 = synth.dims_of(cfg)
    P, R = T * k, d["R"]
    xq_t, xs_t = oracle.mxfp8_quantize(inp["x"])
    xq = np.zeros((P, H), np.uint8)
    xs = np.zeros((P, H // 32), np.uint8)
    xq[:R] = xq_t[d["row_pair"] // k]
    xs[:R] = xs_t[d["row_pair"] // k]
    w = {}
    for key in ("w_gate", "w_up", "w_down"):
        a = inp[key]
        q, s = oracle.mxfp8_quantize(a.reshape(-1, a.shape[-1]))
        w[key] = (q.reshape(a.shape), s.reshape(a.shape[:-1] + (a.shape[-1] // 32,)))
    dw = {key: (dev(q), dev(s)) for key, (q, s) in w.items()}
    y = torch.full((P, H), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = moe.alloc_workspace(moe.moe_expert_ffn_mxfp8_workspace_size(cfg))
    dxq, dxs, off = dev(xq), dev(xs), dev(d["offsets"])
    torch.cuda.synchronize()
    t0 = time.time()
    moe.moe_testing_expert_ffn_mxfp8_stalled(cfg, dxq, dxs, off, dw["w_gate"], dw["w_up"], dw["w_down"], y, ws,
                                             status=st)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    print(f"TIMEOUT mxfp8 ffn: status {int(st.item())} after {elapsed:.2f} s")
    assert int(st.item()) == 6  # MOE_ERR_TIMEOUT
    assert elapsed < 30
    st.zero_()
    moe.moe_expert_ffn_mxfp8(cfg, dxq, dxs, off, dw["w_gate"], dw["w_up"], dw["w_down"], y, ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows = np.arange(R, dtype=np.int64)
    ref = oracle.expert_ffn_mxfp8_rowlist(xq, xs, d["offsets"], w["w_gate"], w["w_up"], w["w_down"], rows)
    err, rms = rel_err(host(y)[:R], ref)
    assert err <= 2e-2 * rms
