"""GPU parity of every step of the hot path against the CPU oracle, on every
seeded workload at its full size, through the C ABI.

Bars: routing indices, counts, offsets, row_pair, pair_row and the x_perm bytes
are bit-exact; routing weights within (k+8)*2^-24 (fp32 expf/sum/divide against
fp64); the expert FFN rows and the layer output within 2e-2 * RMS of the oracle
(bf16 operands, fp32 accumulation, bf16 h, fp32 y); combine within fp32 rounding.
The layer output is checked on every token of every workload except the
16384-token one, where 2048 seeded whole tokens (plus the first and last) are
checked; the expert FFN on at least 2048 grouped rows per workload (every row when
there are fewer), always including the first, middle and last row of every
expert.  Everything else is checked whole.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import OUT_TOL, WEIGHT_TOL, dev, host, inputs, oracle_routing, parity_rows, parity_tokens, rel_err

pytestmark = pytest.mark.gpu

CONFIGS = ["tiny", "decode", "prefill_ep_rank", "skewed", "skewed_rank0", "prefill_full"]
# tokens of the layer output compared with the oracle: all of them, except on the
# 16384-token workload (the oracle would take minutes there)
LAYER_TOKENS = {"prefill_full": 2048}


@pytest.fixture(scope="module")
def moe():
    import torch

    import expert_routing_dispatch_gb300 as m

    assert torch.cuda.is_available()
    m.lib()
    return m


def _zeros(shape, dtype):
    import torch

    return torch.zeros(shape, dtype=dtype, device="cuda")


@pytest.mark.parametrize("name", CONFIGS)
def test_route(moe, name):
    import torch

    cfg, inp = inputs(name)
    T, H, I, E, k, e0, e1 = synth.dims_of(cfg)
    idx = _zeros((T, k), torch.int32)
    w = _zeros((T, k), torch.float32)
    status = _zeros(1, torch.int32)
    moe.moe_route(cfg, dev(inp["logits"]), idx, w, status)
    torch.cuda.synchronize()
    ridx, rw, _ = oracle_routing(name)
    assert int(status.item()) == 0
    assert np.array_equal(host(idx), ridx)
    assert np.abs(host(w).astype(np.float64) - rw).max() <= WEIGHT_TOL(k)


@pytest.mark.parametrize("name", CONFIGS)
def test_dispatch(moe, name):
    import torch

    cfg, inp = inputs(name)
    T, H, I, E, k, e0, e1 = synth.dims_of(cfg)
    n = e1 - e0
    ridx, _, d = oracle_routing(name)
    P = T * k
    counts, offsets = _zeros(n, torch.int32), _zeros(n + 1, torch.int32)
    row_pair = torch.full((P,), -7, dtype=torch.int32, device="cuda")
    pair_row = torch.full((P,), -7, dtype=torch.int32, device="cuda")
    x_perm = _zeros((P, H), torch.int16)
    ws = moe.alloc_workspace(moe.moe_dispatch_workspace_size(cfg))
    moe.moe_dispatch(cfg, dev(inp["x"]), dev(ridx), counts, offsets, row_pair, pair_row, x_perm, ws)
    torch.cuda.synchronize()
    R = d["R"]
    assert np.array_equal(host(counts), d["counts"])
    assert np.array_equal(host(offsets), d["offsets"])
    assert np.array_equal(host(row_pair)[:R], d["row_pair"])
    assert np.array_equal(host(pair_row), d["pair_row"])
    xp = host(x_perm, np.uint16)[:R]
    assert np.array_equal(xp, inp["x"][d["row_pair"] // k])


@pytest.mark.parametrize("name", CONFIGS)
def test_expert_ffn(moe, name):
    import torch

    cfg, inp = inputs(name)
    T, H, I, E, k, e0, e1 = synth.dims_of(cfg)
    _, _, d = oracle_routing(name)
    P, R = T * k, d["R"]
    x_perm = np.zeros((P, H), np.uint16)
    x_perm[:R] = inp["x"][d["row_pair"] // k]  # grouped rows built on the host from the oracle's dispatch
    y_perm = _zeros((P, H), torch.float32)
    status = _zeros(1, torch.int32)
    ws = moe.alloc_workspace(moe.moe_expert_ffn_workspace_size(cfg))
    moe.moe_expert_ffn(cfg, dev(x_perm), dev(d["offsets"]), dev(inp["w_gate"]), dev(inp["w_up"]),
                       dev(inp["w_down"]), y_perm, ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = parity_rows(d["offsets"], at_least=2048)
    if rows.size == 0:
        return
    got = host(y_perm)[rows]
    ref = oracle.expert_ffn_rowlist(x_perm, d["offsets"], inp["w_gate"], inp["w_up"], inp["w_down"], rows)
    err, rms = rel_err(got, ref)
    print(f"PARITY expert_ffn {name} rows {rows.size} of {R}: max|gpu-oracle|/RMS = {err / rms:.3e}")
    assert err <= OUT_TOL * rms, f"max err {err:.3e} vs RMS {rms:.3e} ({err / rms:.2e})"


@pytest.mark.parametrize("name", CONFIGS)
def test_combine(moe, name):
    import torch

    cfg, _ = inputs(name)
    T, H, I, E, k, e0, e1 = synth.dims_of(cfg)
    _, rw, d = oracle_routing(name)
    P = T * k
    y_perm = synth.normal_f32(3, synth.TID_AUX + 9, (P, H))  # synthetic expert outputs
    w32 = rw.astype(np.float32)
    out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    moe.moe_combine(cfg, dev(y_perm), dev(d["pair_row"]), dev(w32), out)
    torch.cuda.synchronize()
    got = host(out)
    ref = oracle.combine_tokens(y_perm, d["pair_row"], w32)
    # fp32 FMA chain vs fp64: |error| <= k * 2^-23 * sum_j |w_j y_j|
    bound = k * 2.0 ** -23 * oracle.combine_tokens(np.abs(y_perm), d["pair_row"], np.abs(w32))
    assert np.all(np.abs(got - ref) <= bound + 1e-30)
    no_local = (d["pair_row"].reshape(T, k) < 0).all(axis=1)
    assert (got[no_local] == 0).all()


@pytest.mark.parametrize("name", CONFIGS)
def test_layer(moe, name):
    import torch

    cfg, inp = inputs(name)
    T, H, I, E, k, e0, e1 = synth.dims_of(cfg)
    out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    idx = _zeros((T, k), torch.int32)
    w = _zeros((T, k), torch.float32)
    status = _zeros(1, torch.int32)
    ws = moe.alloc_workspace(moe.moe_workspace_size(cfg))
    moe.moe_layer(cfg, dev(inp["x"]), dev(inp["logits"]), dev(inp["w_gate"]), dev(inp["w_up"]),
                  dev(inp["w_down"]), out, ws, topk_idx=idx, topk_w=w, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ridx, _, d = oracle_routing(name)
    assert np.array_equal(host(idx), ridx)
    got = host(out)
    no_local = (d["pair_row"].reshape(T, k) < 0).all(axis=1)
    assert (got[no_local] == 0).all()
    toks = parity_tokens(T, LAYER_TOKENS[name]) if name in LAYER_TOKENS else np.arange(T, dtype=np.int64)
    st, ref = oracle.moe_layer_tokens(inp["logits"], inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"], k, e0, e1,
                                      tokens=toks)
    assert st == 0
    err, rms = rel_err(got[toks], ref)
    if rms == 0:
        assert err == 0
    else:
        print(f"PARITY layer {name} tokens {toks.size} of {T}: max|gpu-oracle|/RMS = {err / rms:.3e}")
        assert err <= OUT_TOL * rms, f"max err {err:.3e} vs RMS {rms:.3e} ({err / rms:.2e})"
