"""The seeded input generator: slice-invariance (weights indexed by global expert
id), determinism, and first moments of the distributions (CPU only)."""
import numpy as np

import synth


def test_slices_reproduce_the_full_tensor():
    full = synth.normal_bf16(0, synth.TID_W_GATE, (8, 16, 32), 0.05)
    for e0 in (0, 3, 5):
        part = synth.normal_bf16(0, synth.TID_W_GATE, (2, 16, 32), 0.05, start=e0 * 16 * 32)
        assert np.array_equal(part, full[e0:e0 + 2])
    odd = synth.normal_bf16(0, synth.TID_W_GATE, (7,), 0.05, start=33)
    assert np.array_equal(odd, full.reshape(-1)[33:40])


def test_config_slices_share_weights():
    c_all = synth.config("tiny")
    c_part = synth.config("tiny", e0=4, e1=12)
    wa = synth.make_weights(c_all)
    wp = synth.make_weights(c_part)
    for name in ("w_gate", "w_up", "w_down"):
        assert np.array_equal(wa[name][4:12], wp[name])


def test_deterministic_and_seeded():
    a = synth.normal_f32(0, 2, (1000,))
    b = synth.normal_f32(0, 2, (1000,))
    c = synth.normal_f32(1, 2, (1000,))
    assert np.array_equal(a, b) and not np.array_equal(a, c)


def test_moments():
    a = synth.normal_f32(0, synth.TID_LOGITS, (400000,))
    assert abs(a.mean()) < 0.01 and abs(a.std() - 1) < 0.01
    w = synth.bf16_to_f32(synth.normal_bf16(0, synth.TID_W_UP, (400000,), 0.02))
    assert abs(w.mean()) < 2e-4 and abs(w.std() - 0.02) < 3e-4


def test_bf16_round_to_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0, -0.0], np.float32)
    got = synth.f32_to_bf16(vals)
    # 1+2^-8 is a tie between 1 and 1+2^-7 -> even (1.0); 1+3*2^-8 -> 1+2^-6
    assert got.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x0000, 0x8000]
    assert np.array_equal(synth.bf16_to_f32(got)[:4], np.array([1.0, 1.0, 1.0 + 2 ** -6, -2.5], np.float32))


def test_zipf_bias():
    b = synth.zipf_bias(128)
    assert b[0] == 0.0 and abs(b[31] - 3 * np.log(1 / 32)) < 1e-5
    assert (np.diff(b) < 0).all()
