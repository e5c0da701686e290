"""Pins of the oracle's routing step against brute force, closed forms and
invariants (CPU only).  Routing = top-k of the fp32 expert logits (ties to the
lower expert id), weights = softmax renormalised over the k picks."""
import math

import numpy as np
import pytest

import oracle
import synth


def brute_topk(row, k):
    """Full sort by (-logit, id): an independent definition of the selection."""
    order = sorted(range(len(row)), key=lambda e: (-float(row[e]), e))
    return order[:k]


@pytest.mark.parametrize("E,k", [(5, 1), (5, 3), (8, 8), (16, 4), (33, 7), (128, 8)])
def test_selection_matches_full_sort(E, k):
    rng = np.random.default_rng(E * 100 + k)
    T = 200
    # few distinct values -> many ties; include both signed zeros
    pool = np.array([-1.5, -0.0, 0.0, 0.25, 0.25, 2.0, 7.0], np.float32)
    lg = pool[rng.integers(0, pool.size, size=(T, E))]
    st, idx, _ = oracle.route(lg, k)
    assert st == 0
    for t in range(T):
        assert list(idx[t]) == brute_topk(lg[t], k)


def test_selection_random_normal_full_sort():
    lg = synth.normal_f32(7, synth.TID_AUX, (300, 64))
    st, idx, _ = oracle.route(lg, 6)
    assert st == 0
    for t in range(lg.shape[0]):
        assert list(idx[t]) == brute_topk(lg[t], 6)


def test_signed_zero_ties_to_lower_id():
    lg = np.array([[0.0, -0.0, -1.0], [-0.0, 0.0, -1.0]], np.float32)
    st, idx, w = oracle.route(lg, 1)
    assert st == 0 and idx[:, 0].tolist() == [0, 0]


@pytest.mark.parametrize("k", [1, 2, 4, 8, 16])
def test_all_equal_logits(k):
    lg = np.full((10, 16), 0.3125, np.float32)
    st, idx, w = oracle.route(lg, k)
    assert st == 0
    assert (idx == np.arange(k)[None, :]).all()
    assert (w == 1.0 / k).all()  # exact for k a power of two


def test_k1_weight_is_one():
    lg = synth.normal_f32(1, synth.TID_AUX, (50, 32))
    st, idx, w = oracle.route(lg, 1)
    assert st == 0 and (w == 1.0).all()
    assert (idx[:, 0] == np.argmax(lg, axis=1)).all()


def test_two_expert_closed_form():
    lg = synth.normal_f32(2, synth.TID_AUX, (100, 2), std=3.0)
    st, idx, w = oracle.route(lg, 2)
    assert st == 0
    for t in range(100):
        l0, l1 = float(lg[t, idx[t, 0]]), float(lg[t, idx[t, 1]])
        assert l0 >= l1
        assert abs(w[t, 0] - 1.0 / (1.0 + math.exp(l1 - l0))) < 1e-15
        assert abs(w[t, 1] - 1.0 / (1.0 + math.exp(l0 - l1))) < 1e-15


def test_weights_equal_renormalised_full_softmax():
    lg = synth.normal_f32(3, synth.TID_AUX, (64, 128))
    k = 8
    st, idx, w = oracle.route(lg, k)
    assert st == 0
    for t in range(64):
        p = np.exp(lg[t].astype(np.float64))
        p = p / p.sum()  # softmax over all E experts
        sel = p[idx[t]]
        ref = sel / sel.sum()  # renormalised over the k picks
        assert np.allclose(w[t], ref, rtol=1e-13, atol=0)
        # selection on logits == selection on softmax probabilities (exp monotone)
        assert set(idx[t].tolist()) == set(np.argsort(-p, kind="stable")[:k].tolist())


def test_weights_sum_to_one_and_descend():
    lg = synth.normal_f32(4, synth.TID_AUX, (500, 128))
    st, idx, w = oracle.route(lg, 8)
    assert st == 0
    assert np.all(np.abs(w.sum(axis=1) - 1.0) <= 8 * 2.0 ** -52)
    assert np.all(np.diff(w, axis=1) <= 0)
    assert np.all(np.diff(np.take_along_axis(lg, idx, axis=1), axis=1) <= 0)


def test_hand_worked_example():
    # logits (1, 3, 3, -2, 0.5), k = 3: picks 1, 2 (tie -> lower id first), then 0
    lg = np.array([[1.0, 3.0, 3.0, -2.0, 0.5]], np.float32)
    st, idx, w = oracle.route(lg, 3)
    assert st == 0 and idx[0].tolist() == [1, 2, 0]
    s = 2.0 + math.exp(-2.0)
    assert np.allclose(w[0], [1 / s, 1 / s, math.exp(-2.0) / s], rtol=1e-15)


@pytest.mark.parametrize("bad", [np.nan, np.inf, -np.inf])
def test_nonfinite_logit_is_an_error(bad):
    lg = np.zeros((4, 8), np.float32)
    lg[2, 5] = bad
    st, _, _ = oracle.route(lg, 2)
    assert st == oracle.NONFINITE
