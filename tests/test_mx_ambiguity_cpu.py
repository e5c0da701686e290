"""CPU checks of the MXFP8 rounding-ambiguity helper that the GPU MXFP8 parity
tests use (gpu_helpers.mx_ambiguity / mx_down_bound): values on the E4M3 grid are
never ambiguous, values on a rounding midpoint always are (with the grid spacing
as the allowed change), a block maximum on a power of two makes the block's scale
ambiguous, and the down bound is |W_down| applied to the allowed change."""
import numpy as np

import oracle
from gpu_helpers import e4m3_magnitudes, mx_ambiguity, mx_down_bound


def test_grid_is_the_e4m3_table():
    g = e4m3_magnitudes()
    assert g.size == 127 and g[0] == 0.0 and g[-1] == 448.0 and np.all(np.diff(g) > 0)
    assert g[1] == 2.0 ** -9 and g[8] == 2.0 ** -6 and g[56] == 1.0  # subnormal quantum, smallest normal, 1.0


def test_grid_values_are_unambiguous_and_midpoints_are():
    g = e4m3_magnitudes()
    X = 2.0 ** -3
    # a block whose maximum is 300 * X (scale code 127 - 3 = 124), other entries on the grid or on midpoints
    v = np.array([300.0, 1.0, 1.0625, 0.5 * (1.0 + 1.125), 0.5 * (g[1] + g[2]), 17.0, 96.0, 100.0] + [0.0] * 24)
    h = (v * X)[None, :]
    hs = np.array([[124]], np.uint8)
    amb, delta, samb = mx_ambiguity(h, hs)
    assert not samb.any()
    # 300 is not on the grid (288 / 320) and not near their midpoint 304: unambiguous
    assert list(amb[0, :8]) == [False, False, True, True, True, True, False, True]
    assert delta[0, 2] == 0.125 * X and delta[0, 3] == 0.125 * X and delta[0, 4] == 2.0 ** -9 * X
    assert delta[0, 5] == 2.0 * X and delta[0, 7] == 8.0 * X and (delta[0, ~amb[0]] == 0).all()


def test_block_maximum_on_a_power_of_two_makes_the_scale_ambiguous():
    h = np.zeros((2, 32))
    h[0, :] = np.linspace(-1.0, 1.0, 32) * 0.3
    h[0, 5] = 2.0 ** -2 * 256  # exactly 2^6
    h[1, :] = np.linspace(-1.0, 1.0, 32) * 0.3
    h[1, 5] = 70.0
    hs = np.array([[127 + 6 - 8], [127 + 6 - 8]], np.uint8)
    amb, delta, samb = mx_ambiguity(h, hs)
    assert samb[0, 0] and not samb[1, 0]
    assert amb[0].all()


def test_down_bound_is_abs_weights_times_change():
    rng = np.random.default_rng(0)
    n, H, I = 2, 64, 64
    wq = rng.integers(0, 120, size=(n, H, I)).astype(np.uint8) | (rng.integers(0, 2, size=(n, H, I)) << 7).astype(
        np.uint8)
    ws = np.full((n, H, I // 32), 120, np.uint8)
    offsets = np.array([0, 3, 5], np.int32)
    rows = np.array([0, 2, 3, 4], np.int64)
    dh = np.zeros((4, I))
    dh[1, 7] = 0.5
    dh[3, 0] = 2.0
    b = mx_down_bound(rows, offsets, (wq, ws), dh)
    W0 = np.abs(oracle.mxfp8_dequantize(wq[0], ws[0]))
    W1 = np.abs(oracle.mxfp8_dequantize(wq[1], ws[1]))
    assert np.allclose(b[1], 0.5 * W0[:, 7]) and np.allclose(b[3], 2.0 * W1[:, 0])
    assert (b[0] == 0).all() and (b[2] == 0).all()
