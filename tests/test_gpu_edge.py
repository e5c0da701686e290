"""GPU edge cases against the oracle, through the C ABI: T=1, k=1, k=E, E not a
multiple of 32, ragged H/I tails, empty local range (R=0), all-tied logits,
non-finite logits (device status), one token per expert, the largest E and k,
determinism, and range decomposition (four local ranges sum to the full range).

Routing is bit-exact.  Layer outputs on these off-workload shapes are held to the
elementwise bound that rounding h to bf16 implies (see gpu_helpers.bf16_h_bound);
the six workloads themselves are held to 2e-2 * RMS in test_gpu_parity."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import WEIGHT_TOL, bf16_h_bound, dev, host, inputs, rel_err, sample_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import torch

    import expert_routing_dispatch_gb300 as m

    assert torch.cuda.is_available()
    m.lib()
    return m


def small_inputs(T, H, I, E, k, e0, e1, seed=0, w_std=0.05, logits=None):
    x = synth.normal_bf16(seed, synth.TID_X, (T, H), 1.0)
    lg = synth.normal_f32(seed, synth.TID_LOGITS, (T, E)) if logits is None else logits
    n = e1 - e0
    wg = synth.normal_bf16(seed, synth.TID_W_GATE, (n, I, H), w_std, start=e0 * I * H)
    wu = synth.normal_bf16(seed, synth.TID_W_UP, (n, I, H), w_std, start=e0 * I * H)
    wd = synth.normal_bf16(seed, synth.TID_W_DOWN, (n, H, I), w_std, start=e0 * H * I)
    return dict(x=x, logits=lg, w_gate=wg, w_up=wu, w_down=wd)


def tup(d):
    return tuple(getattr(d, f) for f in ("T", "H", "I", "E", "k", "e0", "e1"))


def run_layer(moe, dims, inp, want_status=0):
    import torch

    T, H, I, E, k, e0, e1 = tup(dims)
    out = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = moe.alloc_workspace(moe.moe_workspace_size(dims))
    moe.moe_layer(dims, dev(inp["x"]), dev(inp["logits"]), dev(inp["w_gate"]), dev(inp["w_up"]),
                  dev(inp["w_down"]), out, ws, topk_idx=idx, topk_w=w, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == want_status
    return host(out), host(idx), host(w)


def check_layer(moe, dims, inp, tokens=None):
    T, H, I, E, k, e0, e1 = tup(dims)
    out, idx, w = run_layer(moe, dims, inp)
    st, ridx, rw = oracle.route(inp["logits"], k)
    assert st == 0
    assert np.array_equal(idx, ridx)
    assert np.abs(w.astype(np.float64) - rw).max() <= WEIGHT_TOL(k)
    toks = np.arange(T) if tokens is None else tokens
    st, ref = oracle.moe_layer_tokens(inp["logits"], inp["x"], inp["w_gate"], inp["w_up"], inp["w_down"], k, e0, e1,
                                      tokens=toks)
    # these shapes lie outside the six workloads: the bar is the elementwise bound
    # implied by rounding h to bf16 (k = 1 has no averaging over slots)
    bound = bf16_h_bound(inp, k, e0, e1, toks, ridx, rw) + 1e-6 * np.abs(ref).max()
    diff = np.abs(out[toks].astype(np.float64) - ref)
    err, rms = rel_err(out[toks], ref)
    print(f"EDGE {tup(dims)} max|gpu-oracle|/RMS = {err / max(rms, 1e-300):.3e}, "
          f"max err/bound = {(diff / bound).max():.3f}")
    assert np.all(diff <= bound)
    return out


@pytest.mark.parametrize("dims", [
    (1, 64, 64, 4, 1, 0, 4),          # T=1, k=1
    (1, 256, 128, 8, 8, 0, 8),        # T=1, k=E
    (37, 128, 64, 8, 8, 2, 5),        # k=E, partial range
    (300, 320, 192, 6, 2, 0, 6),      # ragged H (256+64) and I (128+64) tails, several m-tiles
    (200, 192, 320, 40, 5, 7, 33),    # E not a multiple of 32
    (513, 256, 128, 3, 1, 1, 2),      # single local expert, m-tile tails
])
def test_layer_small_shapes(moe, dims):
    inp = small_inputs(*dims)
    check_layer(moe, moe.Dims(*dims), inp)


# The same kinds of edges above the fused threshold (T*k > 8192 pairs), so they run
# the split kernels: ragged H / I tails (a partial last weight tile in both GEMMs),
# E not a multiple of 32 with a partial range, a single local expert with an m-tile
# tail, and k = E.  The oracle checks a sample of tokens (all of them when small).
@pytest.mark.parametrize("dims", [
    (4200, 320, 192, 6, 2, 0, 6),     # ragged H (256+64) and I (128+64) tails
    (2000, 192, 320, 40, 5, 7, 33),   # E not a multiple of 32, partial range, I = 2.5 gate/up tiles
    (9000, 256, 128, 3, 1, 1, 2),     # single local expert, 9000 rows = 70 m-tiles + 40
    (1100, 448, 704, 8, 8, 2, 5),     # k = E, partial range, H = 1.75 down tiles, I = 5.5 gate/up tiles
])
def test_layer_small_shapes_split_path(moe, dims):
    T, k = dims[0], dims[4]
    assert T * k > moe.FUSED_MAX_PAIRS
    inp = small_inputs(*dims)
    toks = None if T <= 2000 else np.unique(np.r_[np.arange(0, T, 7), T - 1])
    check_layer(moe, moe.Dims(*dims), inp, tokens=toks)


def test_empty_local_range(moe):
    # all-equal logits: every token picks experts 0..3, so [8, 16) receives nothing (R = 0)
    T, H, I, E, k, e0, e1 = dims = (64, 256, 128, 16, 4, 8, 16)
    inp = small_inputs(*dims, logits=np.zeros((T, E), np.float32))
    out, idx, w = run_layer(moe, moe.Dims(*dims), inp)
    assert (out == 0).all()
    assert (idx == np.arange(k)[None, :]).all() and (w == 0.25).all()


def test_all_ties_routing(moe):
    import torch

    T, E, k = 50, 64, 8
    d = moe.Dims(T, 64, 64, E, k, 0, E)
    lg = np.full((T, E), -1.25, np.float32)
    lg[::2, 40:] = -0.0  # signed zeros tie with each other (and beat -1.25)
    lg[1::2, :30] = 0.0
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    moe.moe_route(d, dev(lg), idx, w)
    torch.cuda.synchronize()
    st, ridx, rw = oracle.route(lg, k)
    assert np.array_equal(host(idx), ridx)
    assert (host(w) == 0.125).all()


@pytest.mark.parametrize("bad", [np.nan, np.inf, -np.inf])
def test_nonfinite_logits_set_status(moe, bad):
    T, H, I, E, k, e0, e1 = dims = (40, 128, 64, 16, 4, 0, 16)
    lg = synth.normal_f32(0, synth.TID_LOGITS, (T, E))
    lg[7, 3] = bad
    inp = small_inputs(*dims, logits=lg)
    out, idx, _ = run_layer(moe, moe.Dims(*dims), inp, want_status=5)
    assert ((idx >= 0) & (idx < E)).all()  # outputs undefined, but every index stays in bounds


def test_largest_E_and_k_routing(moe):
    import torch

    T, E, k = 300, 1024, 32
    lg = synth.normal_f32(4, synth.TID_LOGITS, (T, E))
    lg[:, 500:520] = 1.5  # a block of ties inside the top-k
    d = moe.Dims(T, 64, 64, E, k, 0, E)
    idx = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    moe.moe_route(d, dev(lg), idx, w)
    torch.cuda.synchronize()
    st, ridx, rw = oracle.route(lg, k)
    assert np.array_equal(host(idx), ridx)
    assert np.abs(host(w).astype(np.float64) - rw).max() <= WEIGHT_TOL(k)


def test_one_token_per_expert(moe):
    # "all experts activated with a single token" (MoE GEMM section): T = E = 128,
    # token t's top-1 is expert t; full-size expert weights of the decode workload
    cfg, inp = inputs("decode")
    T, H, I, E, k, e0, e1 = 128, cfg["H"], cfg["I"], 128, 1, 0, 128
    lg = synth.normal_f32(1, synth.TID_LOGITS, (T, E))
    lg[np.arange(T), np.arange(T)] += 20.0
    x = synth.normal_bf16(1, synth.TID_X, (T, H), 1.0)
    sub = dict(x=x, logits=lg, w_gate=inp["w_gate"], w_up=inp["w_up"], w_down=inp["w_down"])
    check_layer(moe, moe.Dims(T, H, I, E, k, e0, e1), sub, tokens=sample_tokens(T, 16))


def test_deterministic(moe):
    cfg, inp = inputs("prefill_ep_rank")
    dims = moe.Dims.of(cfg)
    a, ia, wa = run_layer(moe, dims, inp)
    b, ib, wb = run_layer(moe, dims, inp)
    assert np.array_equal(ia, ib) and np.array_equal(wa, wb)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_range_decomposition_full_size(moe):
    cfg, inp = inputs("prefill_full")
    T, H, I, E, k, e0, e1 = synth.dims_of(cfg)
    full, _, _ = run_layer(moe, moe.Dims.of(cfg), inp)
    acc = np.zeros_like(full, dtype=np.float64)
    for lo in range(0, E, 32):
        part_inp = dict(inp)
        for nme in ("w_gate", "w_up", "w_down"):
            part_inp[nme] = inp[nme][lo:lo + 32]
        part, _, _ = run_layer(moe, moe.Dims(T, H, I, E, k, lo, lo + 32), part_inp)
        acc += part
    rms = float(np.sqrt((full.astype(np.float64) ** 2).mean()))
    # same bf16 expert rows in both; only the fp32 summation order differs
    assert np.abs(acc - full).max() <= 1e-4 * rms
