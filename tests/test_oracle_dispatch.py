"""Pins of the oracle's dispatch step (select the pairs routed to the local
expert range, count, prefix offsets, stable permutation) -- CPU only."""
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def check_dispatch(idx, e0, e1, d):
    T, k = idx.shape
    n = e1 - e0
    flat = idx.reshape(-1)
    inr = (flat >= e0) & (flat < e1)
    R = int(inr.sum())
    # counts by an independent histogram
    assert (d["counts"] == np.bincount(flat[inr] - e0, minlength=n)).all()
    assert d["R"] == R and d["offsets"][-1] == R and d["offsets"][0] == 0
    assert (np.diff(d["offsets"]) == d["counts"]).all()
    # permutation = stable sort of the in-range pairs by expert (numpy's stable argsort)
    pairs = np.nonzero(inr)[0]
    ref = pairs[np.argsort(flat[pairs], kind="stable")]
    assert (d["row_pair"] == ref).all()
    # bijection and inverse
    pr = d["pair_row"]
    assert (pr[~inr] == -1).all()
    assert (pr[d["row_pair"]] == np.arange(R)).all()
    # each group ascending, and every row belongs to its expert
    for e in range(n):
        rows = d["row_pair"][d["offsets"][e]:d["offsets"][e + 1]]
        assert (np.diff(rows) > 0).all()
        assert (flat[rows] == e0 + e).all()


@pytest.mark.parametrize("E,k,e0,e1", [(16, 4, 0, 16), (16, 4, 3, 11), (128, 8, 0, 32), (128, 8, 96, 128), (7, 7, 2, 3)])
def test_dispatch_invariants(E, k, e0, e1):
    lg = synth.normal_f32(11, synth.TID_AUX, (333, E))
    st, idx, _ = oracle.route(lg, k)
    assert st == 0
    check_dispatch(idx, e0, e1, oracle.dispatch(idx, e0, e1))


def test_empty_local_range():
    # all-equal logits: every token picks experts 0..k-1, so [8, 16) receives nothing
    lg = np.zeros((50, 16), np.float32)
    st, idx, _ = oracle.route(lg, 4)
    d = oracle.dispatch(idx, 8, 16)
    assert d["R"] == 0 and (d["counts"] == 0).all() and (d["pair_row"] == -1).all()
    d = oracle.dispatch(idx, 0, 8)
    assert d["R"] == 200 and d["counts"].tolist() == [50, 50, 50, 50, 0, 0, 0, 0]
    check_dispatch(idx, 0, 8, d)


def test_tokens_per_expert_worked_example():
    """Mean load per expert T*k/E ("Prefillers" section: 6000*8/128 = 375)."""
    with open(os.path.join(GOLDEN, "tokens_per_expert.txt")) as f:
        T, k, E, per = [int(v) for v in next(l for l in f if not l.startswith("#")).split()]
    assert T * k // E == per and T * k % E == 0
    lg = synth.normal_f32(0, synth.TID_LOGITS, (T, E))
    st, idx, _ = oracle.route(lg, k)
    d = oracle.dispatch(idx, 0, E)
    assert d["counts"].sum() == T * k
    assert d["counts"].mean() == per  # exact: every pair lands on some expert
    # i.i.d. logits -> each count ~ Binomial(T, k/E): std sqrt(T*k/E*(1-k/E)) ~ 18.8
    sd = (T * k / E * (1 - k / E)) ** 0.5
    assert abs(d["counts"].std() - sd) < 0.35 * sd
    assert d["counts"].min() > per - 6 * sd and d["counts"].max() < per + 6 * sd


def test_range_slices_partition_pairs():
    lg = synth.normal_f32(5, synth.TID_AUX, (1000, 128))
    st, idx, _ = oracle.route(lg, 8)
    full = oracle.dispatch(idx, 0, 128)
    seen = np.zeros(idx.size, np.int32)
    for e0 in range(0, 128, 32):
        d = oracle.dispatch(idx, e0, e0 + 32)
        seen[d["row_pair"]] += 1
        assert (d["counts"] == full["counts"][e0:e0 + 32]).all()
    assert (seen == 1).all()


def test_one_token_per_expert_workloads():
    """'MoE GEMM' section: every local expert receives exactly one token."""
    for ep in (1, 8, 32):
        cfg = synth.config(f"one_token_per_expert_ep{ep}")
        lg = synth.make_logits(cfg)
        st, idx, w = oracle.route(lg, cfg["k"])
        d = oracle.dispatch(idx, cfg["e0"], cfg["e1"])
        assert st == 0 and (d["counts"] == 1).all() and d["R"] == cfg["T"] == 128 // ep
        assert (w == 1.0).all()
