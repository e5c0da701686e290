"""moe_combine_accumulate: the accumulation step of DP-EP ("Data Parallel and
Expert Parallel" section: expert results return to the tokens' source rank and
are accumulated there), emulated on one GPU by accumulating the contributions of
several expert ranges into one output buffer.  Checked against the oracle's
combine over the full range, within the fp32 summation bound."""
import numpy as np
import pytest

import oracle
import synth
from gpu_helpers import dev, host, oracle_routing, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import torch

    import expert_routing_dispatch_gb300 as m

    assert torch.cuda.is_available()
    m.lib()
    return m


@pytest.mark.parametrize("name,parts", [("decode", 2), ("decode", 4), ("prefill_full", 4)])
def test_accumulating_expert_ranges_equals_full_combine(moe, name, parts):
    import torch

    cfg, _ = inputs(name)
    T, H, I, E, k, e0, e1 = synth.dims_of(cfg)
    idx, w64, d = oracle_routing(name)
    P = T * k
    y_perm = synth.normal_f32(5, synth.TID_AUX + 10, (P, H))  # synthetic expert outputs
    w32 = w64.astype(np.float32)
    flat_e = idx.reshape(-1)
    out = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    first = None
    width = (e1 - e0) // parts
    for q in range(parts):
        lo, hi = e0 + q * width, e0 + (q + 1) * width
        pr = np.where((flat_e >= lo) & (flat_e < hi), d["pair_row"], -1).astype(np.int32)
        moe.moe_combine_accumulate(cfg, dev(y_perm), dev(pr), dev(w32), out)
        if q == 0:  # accumulating onto zeros is the plain combine, bit for bit
            torch.cuda.synchronize()
            first = host(out).copy()
            plain = torch.full((T, H), float("nan"), dtype=torch.float32, device="cuda")
            moe.moe_combine(cfg, dev(y_perm), dev(pr), dev(w32), plain)
            torch.cuda.synchronize()
            assert np.array_equal(first.view(np.uint32), host(plain).view(np.uint32))
    torch.cuda.synchronize()
    got = host(out)
    ref = oracle.combine_tokens(y_perm, d["pair_row"], w32)
    # fp32 FMA chains per range plus the running additions: |err| <= (k + parts) * 2^-23 * sum_j |w_j y_j|
    bound = (k + parts) * 2.0 ** -23 * oracle.combine_tokens(np.abs(y_perm), d["pair_row"], np.abs(w32))
    assert np.all(np.abs(got - ref) <= bound + 1e-30)
