"""More shapes and usage patterns through the C ABI, against the oracle: the
largest E and k on both paths, a DeepSeek-like H=7168 / I=2048 layer on both
paths, the fused launch's determinism, a non-default CUDA stream, and one large
workspace reused across problems of different sizes.  Off-workload shapes are
held to the elementwise bf16-h rounding bound (see gpu_helpers.bf16_h_bound)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import bf16_h_bound, dev, host, rel_err, sample_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import torch

    import expert_routing_dispatch_gb300 as m

    assert torch.cuda.is_available()
    m.lib()
    return m


def make(T, H, I, E, k, e0, e1, seed=11, w_std=0.03):
    n = e1 - e0
    return dict(x=synth.normal_bf16(seed, synth.TID_X, (T, H), 1.0),
                logits=synth.normal_f32(seed, synth.TID_LOGITS, (T, E)),
                w_gate=synth.normal_bf16(seed, synth.TID_W_GATE, (n, I, H), w_std, start=e0 * I * H),
                w_up=synth.normal_bf16(seed, synth.TID_W_UP, (n, I, H), w_std, start=e0 * I * H),
                w_down=synth.normal_bf16(seed, synth.TID_W_DOWN, (n, H, I), w_std, start=e0 * H * I))


def run(moe, dims, inp, ws=None, stream=None):
    import torch

    T, H, k = dims.T, dims.H, dims.k
    out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    if ws is None:
        ws = moe.alloc_workspace(moe.moe_workspace_size(dims))
    args = [dev(inp[n]) for n in ("x", "logits", "w_gate", "w_up", "w_down")]
    if stream is not None:
        with torch.cuda.stream(stream):
            moe.moe_layer(dims, *args, out, ws, topk_idx=idx, status=st, stream=stream)
    else:
        moe.moe_layer(dims, *args, out, ws, topk_idx=idx, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return host(out), host(idx)


def check(moe, dims, inp, ntok=48):
    T, k, e0, e1 = dims.T, dims.k, dims.e0, dims.e1
    out, idx = run(moe, dims, inp)
    st, ridx, rw = oracle.route(inp["logits"], k)
    assert st == 0 and np.array_equal(idx, ridx)
    toks = sample_tokens(T, ntok)
    st, ref = oracle.moe_layer_tokens(inp["logits"], inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"], k, e0, e1,
                                      tokens=toks)
    bound = bf16_h_bound(inp, k, e0, e1, toks, ridx, rw) + 1e-6 * np.abs(ref).max()
    diff = np.abs(out[toks].astype(np.float64) - ref)
    err, rms = rel_err(out[toks], ref)
    print(f"SHAPE T={T} H={dims.H} I={dims.I} E={dims.E} k={k} [{e0},{e1}) max/RMS={err / rms:.3e} "
          f"max err/bound={(diff / bound).max():.3f}")
    assert np.all(diff <= bound)
    return out


@pytest.mark.parametrize("T", [64, 300])  # 64*32 pairs run fused, 300*32 = 9600 run split
def test_largest_E_and_k(moe, T):
    dims = moe.Dims(T, 128, 128, 1024, 32, 100, 612)
    check(moe, dims, make(T, 128, 128, 1024, 32, 100, 612))


@pytest.mark.parametrize("T,k", [(200, 6), (1500, 6)])  # 1200 pairs fused, 9000 split
def test_deepseek_like_shape(moe, T, k):
    H, I, E, e0, e1 = 7168, 2048, 64, 8, 24
    check(moe, moe.Dims(T, H, I, E, k, e0, e1), make(T, H, I, E, k, e0, e1, w_std=0.02), ntok=24)


def test_fused_launch_deterministic(moe):
    cfg = synth.config("decode")
    inp = synth.make_inputs(cfg)
    dims = moe.Dims.of(cfg)
    a, _ = run(moe, dims, inp)
    b, _ = run(moe, dims, inp)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_non_default_stream_and_reused_workspace(moe):
    import torch

    s = torch.cuda.Stream()
    big = moe.Dims(2000, 256, 192, 32, 4, 0, 32)
    ws = moe.alloc_workspace(moe.moe_workspace_size(big))
    for dims in (big, moe.Dims(50, 256, 192, 32, 4, 8, 24), moe.Dims(2000, 256, 192, 32, 4, 16, 32)):
        inp = make(dims.T, dims.H, dims.I, dims.E, dims.k, dims.e0, dims.e1)
        a, _ = run(moe, dims, inp, ws=ws, stream=s)
        b, _ = run(moe, dims, inp)  # fresh workspace, current stream
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
