"""moe_dispatch_noalloc: the dispatch entry point for callers that cannot
allocate device memory (a plug-in whose host runtime owns all device buffers
and gives it no allocator, or a serving loop that forbids cudaMalloc because it
can synchronise the device).  Its scratch is a fixed array inside libmoe.

Checked through the C ABI against moe_dispatch (which takes a caller-allocated
workspace): every output must match bit for bit -- dispatch is integer and byte
work -- on two calls in a row with different problems, so that stale contents
left in the shared array by the first call would show up in the second.  This
file is named to be collected last, and passes alone or after the other tests.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import torch

    import expert_routing_dispatch_gb300 as m

    assert torch.cuda.is_available()
    m.lib()
    return m


def _dispatch_both(moe, cfg):
    import torch

    T, H, I, E, k, e0, e1 = synth.dims_of(cfg)
    n, P = e1 - e0, T * k
    inp = synth.make_inputs(cfg, weights=False)
    st, idx, _ = oracle.route(inp["logits"], k)
    assert st == 0
    x = torch.from_numpy(inp["x"].view(np.int16)).cuda()
    topk = torch.from_numpy(idx).cuda()

    def outputs():
        return dict(counts=torch.full((n,), -3, dtype=torch.int32, device="cuda"),
                    offsets=torch.full((n + 1,), -3, dtype=torch.int32, device="cuda"),
                    row_pair=torch.full((P,), -3, dtype=torch.int32, device="cuda"),
                    pair_row=torch.full((P,), -3, dtype=torch.int32, device="cuda"),
                    x_perm=torch.zeros((P, H), dtype=torch.int16, device="cuda"))

    ref, got = outputs(), outputs()
    ws = moe.alloc_workspace(moe.moe_dispatch_workspace_size(cfg))
    moe.moe_dispatch(cfg, x, topk, ref["counts"], ref["offsets"], ref["row_pair"], ref["pair_row"], ref["x_perm"], ws)
    moe.moe_dispatch_noalloc(cfg, x, topk, got["counts"], got["offsets"], got["row_pair"], got["pair_row"],
                             got["x_perm"])
    torch.cuda.synchronize()
    R = int(ref["offsets"][-1].item())
    for name in ("counts", "offsets", "pair_row"):
        assert torch.equal(ref[name], got[name]), name
    assert torch.equal(ref["row_pair"][:R], got["row_pair"][:R])
    assert torch.equal(ref["x_perm"][:R], got["x_perm"][:R])
    return R


def test_noalloc_dispatch_matches_dispatch_on_two_calls_in_a_row(moe):
    # first the 16384-token workload (64 chunks x 128 experts = 8192 of the array's
    # 262144 entries), then a smaller one with a different local range: leftovers
    # from the first call must not leak
    r1 = _dispatch_both(moe, synth.config("prefill_full"))
    r2 = _dispatch_both(moe, synth.config("skewed_rank0"))
    assert r1 == 16384 * 8 and r2 > 0


def test_noalloc_dispatch_at_the_size_limit_then_a_small_call(moe):
    # T*k = 4,194,304 pairs over 128 local experts: 2048 chunks x 128 = 262144
    # entries, the whole array; then a small problem on a partial range
    big = synth.config("prefill_full", T=1 << 19, H=64)
    assert -(-big["T"] * big["k"] // 2048) * (big["e1"] - big["e0"]) == 1 << 18
    r1 = _dispatch_both(moe, big)
    r2 = _dispatch_both(moe, synth.config("tiny", e0=3, e1=11))
    assert r1 == (1 << 19) * 8 and r2 > 0


def test_noalloc_rejects_problems_beyond_its_fixed_scratch(moe):
    # ceil(T*k / 2048) * n > 262144: refused on the host, nothing launched
    d = moe.Dims(1 << 20, 64, 64, 1024, 8, 0, 1024)
    ok = 1 << 20  # aligned, never dereferenced
    st = moe.lib().moe_dispatch_noalloc(ctypes.byref(d), ok, ok, ok, ok, ok, ok, ok, None)
    assert st == 2  # MOE_ERR_UNSUPPORTED
