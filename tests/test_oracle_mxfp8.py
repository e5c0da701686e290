"""Pins of the oracle's MXFP8 path (the "MoE GEMM" section of "Hosting Qwen on
Blackwell" deploys MXFP8 expert GEMMs; the format is read as OCP MX v1.0 MXFP8:
E4M3 elements, one UE8M0 scale per 32 elements) -- CPU only.

- E4M3 values against the specification's table (tests/golden/e4m3_values.txt)
- each element code is the nearest finite E4M3 value of v / X (ties to an even
  mantissa, saturating at 448), checked by exhaustive search over all codes
- the scale code in closed form: floor(log2(amax)) - 8 + 127, 0 for a zero block,
  with amax the largest magnitude of either sign (mirrored blocks share the scale)
- the MX expert FFN against a float64 evaluation of the dequantised operands,
  and against the (separately pinned) bf16 oracle within the bound that
  quantising h implies
"""
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32_to_bf16_bits(v):
    return synth.f32_to_bf16(np.asarray(v, np.float32))


def quant(values):
    """quantise float values exactly representable in bf16, one row"""
    a = f32_to_bf16_bits(np.asarray(values, np.float32)).reshape(1, -1)
    assert np.array_equal(synth.bf16_to_f32(a).ravel(), np.asarray(values, np.float32))
    return oracle.mxfp8_quantize(a)


def test_e4m3_table_values():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e4m3_values.txt")) if not l.startswith("#") and l.strip()]
    for code_s, val_s in rows:
        code, val = int(code_s, 16), float(val_s)
        # a block whose amax is 448 has scale 2^0 (code 127): dequantising `code` gives the element value
        q = np.full((1, 32), code, np.uint8)
        s = np.full((1, 1), 127, np.uint8)
        got = oracle.mxfp8_dequantize(q, s)[0, 0]
        assert got == val and math.copysign(1.0, got) == math.copysign(1.0, val), (code_s, got, val)


def _all_finite_codes():
    codes = [c for c in range(256) if (c & 0x7F) != 0x7F]
    vals = oracle.mxfp8_dequantize(np.array([codes[:128], codes[128:] + [0] * (256 - len(codes))], np.uint8)[:, :len(codes[:128])],
                                   np.full((2, 4), 127, np.uint8))
    return codes, np.concatenate([vals[0], vals[1][: len(codes) - 128]])


def test_nearest_code_by_exhaustive_search():
    codes, vals = _all_finite_codes()
    rng = np.random.default_rng(7)
    for trial in range(200):
        scale = rng.uniform(-12, 12)
        block = (rng.standard_normal(32) * 2.0 ** scale).astype(np.float32)
        block = synth.bf16_to_f32(f32_to_bf16_bits(block))  # bf16-exact inputs
        q, s = oracle.mxfp8_quantize(f32_to_bf16_bits(block).reshape(1, 32))
        x = 2.0 ** (int(s[0, 0]) - 127)
        for v, c in zip(block.astype(np.float64), q[0]):
            t = v / x
            d = np.abs(vals - t)
            best = d.min()
            cand = [codes[i] for i in np.nonzero(d == best)[0]]
            if abs(t) >= 448:
                cand = [0x7E | (0x80 if t < 0 else 0)]
            elif len(cand) > 1:  # a tie: the even mantissa (same sign as t)
                cand = [cc for cc in cand if (cc & 1) == 0 and ((cc & 0x80) != 0) == (t < 0 or (t == 0 and math.copysign(1, t) < 0))]
            assert c in cand or (best == 0 and vals[codes.index(c)] == 0), (v, t, c, cand)


def test_subnormal_codes_by_exhaustive_search():
    # amax 448 gives X = 2^0, so the other elements are encoded as they are: quarter steps
    # of the subnormal quantum 2^-9 (exact codes, ties and in-between values), both signs
    codes, vals = _all_finite_codes()
    for sign in (1.0, -1.0):
        elems = [sign * j * 2.0 ** -11 for j in range(1, 32)]
        q, s = quant([448.0] + elems)
        assert s[0, 0] == 127
        for t, c in zip(elems, q[0, 1:]):
            d = np.abs(vals - t)
            cand = [codes[i] for i in np.nonzero(d == d.min())[0]]
            if len(cand) > 1:  # a tie: the even mantissa, with the sign of t
                cand = [cc for cc in cand if (cc & 1) == 0 and ((cc & 0x80) != 0) == (t < 0)]
            assert c in cand or (vals[codes.index(c)] == 0 and d.min() == abs(t) and 0.0 in [vals[codes.index(cc)] for cc in cand]), (t, c, cand)


def test_scale_code_closed_form():
    for p in range(-20, 21, 3):
        for f in (1.0, 1.25, 1.75, 1.9921875):
            amax = f * 2.0**p
            q, s = quant([amax] + [0.0] * 31)
            assert s[0, 0] == p - 8 + 127
            # amax / X = f * 2^8: exact below 448, saturating above
            want = min(f * 256.0, 448.0)
            assert oracle.mxfp8_dequantize(q, s)[0, 0] == want * 2.0 ** (p - 8)
    q, s = quant([0.0] * 32)
    assert s[0, 0] == 0 and (q == 0).all()


def test_scale_follows_largest_magnitude_of_either_sign():
    # OCP MX: the shared scale comes from max |v| over the block, so mirroring a block
    # (v -> -v) keeps its scale code and flips only the sign bit of every element code
    rng = np.random.default_rng(11)
    for trial in range(50):
        block = (rng.standard_normal(32) * 2.0 ** rng.uniform(-12, 12)).astype(np.float32)
        bits = f32_to_bf16_bits(block).reshape(1, 32)
        q, s = oracle.mxfp8_quantize(bits)
        qn, sn = oracle.mxfp8_quantize(bits ^ np.uint16(0x8000))
        assert np.array_equal(sn, s)
        assert np.array_equal(qn, q ^ np.uint8(0x80))
    # a block whose largest magnitude is negative: floor(log2 3) = 1, X = 2^-7, all exact
    q, s = quant([-3.0, 1.0, 0.5] + [0.0] * 29)
    assert s[0, 0] == 1 - 8 + 127
    assert list(oracle.mxfp8_dequantize(q, s)[0, :3]) == [-3.0, 1.0, 0.5]


def test_ties_signed_zero_and_saturation():
    # X = 2^0 (amax 256..511): 17 lies between 16 and 18 (step 2 in [16, 32)) -> 16 (even)
    q, s = quant([256.0, 17.0, 19.0, -17.0, -(2.0 ** -100), 500.0] + [0.0] * 26)
    d = oracle.mxfp8_dequantize(q, s)[0]
    assert s[0, 0] == 127
    assert d[1] == 16.0 and d[2] == 20.0 and d[3] == -16.0
    assert q[0, 4] == 0x80  # a negative value that rounds to zero keeps its sign
    assert d[5] == 448.0  # 500 saturates


@pytest.mark.parametrize("H,I,n", [(64, 32, 2), (96, 64, 3)])
def test_mx_ffn_against_dequantised_float64(H, I, n):
    rng = np.random.default_rng(H + I)
    R = 7
    x = f32_to_bf16_bits(rng.standard_normal((R, H)).astype(np.float32))
    wg = f32_to_bf16_bits((rng.standard_normal((n * I, H)) * 0.1).astype(np.float32))
    wu = f32_to_bf16_bits((rng.standard_normal((n * I, H)) * 0.1).astype(np.float32))
    wd = f32_to_bf16_bits((rng.standard_normal((n * H, I)) * 0.1).astype(np.float32))
    xq, xs = oracle.mxfp8_quantize(x)
    g = [oracle.mxfp8_quantize(w) for w in (wg, wu, wd)]
    offsets = np.array([0, 3, 5, 7][: n + 1] if n == 3 else [0, 4, 7], np.int32)
    rows = np.arange(R, dtype=np.int64)
    shape = lambda pair, a, b: (pair[0].reshape(n, a, b), pair[1].reshape(n, a, b // 32))
    y, h, hq, hs = oracle.expert_ffn_mxfp8_rowlist(xq, xs, offsets, shape(g[0], I, H), shape(g[1], I, H),
                                                   shape(g[2], H, I), rows, want_h=True)
    X = oracle.mxfp8_dequantize(xq, xs)
    G, U, D = (oracle.mxfp8_dequantize(*p) for p in g)
    for r in range(R):
        e = int(np.searchsorted(offsets, r, side="right") - 1)
        gg = G[e * I:(e + 1) * I] @ X[r]
        uu = U[e * I:(e + 1) * I] @ X[r]
        hh = gg / (1.0 + np.exp(-gg)) * uu
        assert np.allclose(h[r], hh, rtol=1e-12, atol=1e-12)
        # h is quantised by the (pinned) quantiser; y is the dequantised down GEMM
        hdq = oracle.mxfp8_dequantize(hq[r:r + 1], hs[r:r + 1])[0]
        assert np.allclose(y[r], D[e * H:(e + 1) * H] @ hdq, rtol=1e-12, atol=1e-12)
    # h_in replaces the down GEMM's operand
    y2 = oracle.expert_ffn_mxfp8_rowlist(xq, xs, offsets, shape(g[0], I, H), shape(g[1], I, H), shape(g[2], H, I),
                                         rows, h_in=(np.zeros_like(hq), np.zeros_like(hs)))
    assert (y2 == 0).all()


def test_mx_ffn_near_bf16_oracle_when_operands_are_exact():
    """Operands that MXFP8 represents exactly (bf16 values k/8 with |k| <= 14 and a
    block max of 1.75 -> scale 2^-8, elements 32k <= 448): the MX path then differs from the bf16
    oracle only by the quantisation of h, |dy_j| <= sum_i |Wd_ji| |h_i - hq_i|."""
    rng = np.random.default_rng(3)
    H, I, n, R = 64, 64, 1, 5
    mk = lambda shape: f32_to_bf16_bits((rng.integers(-14, 15, shape) / 8.0).astype(np.float32))
    x, wg, wu, wd = mk((R, H)), mk((I, H)), mk((I, H)), mk((H, I))
    for blk in (x, wg, wu, wd):
        blk[:, ::32] = f32_to_bf16_bits(np.float32(1.75))  # every block's amax is 1.75
    q = [oracle.mxfp8_quantize(a) for a in (x, wg, wu, wd)]
    for a, (qq, ss) in zip((x, wg, wu, wd), q):
        assert np.array_equal(oracle.mxfp8_dequantize(qq, ss), synth.bf16_to_f32(a).astype(np.float64))
    offsets = np.array([0, R], np.int32)
    rows = np.arange(R, dtype=np.int64)
    y, h, hq, hs = oracle.expert_ffn_mxfp8_rowlist(q[0][0], q[0][1], offsets, (q[1][0][None], q[1][1][None]),
                                                   (q[2][0][None], q[2][1][None]), (q[3][0][None], q[3][1][None]),
                                                   rows, want_h=True)
    ref = oracle.expert_ffn_rows(x, offsets, wg[None], wu[None], wd[None])
    dh = np.abs(h - oracle.mxfp8_dequantize(hq, hs))
    bound = dh @ np.abs(synth.bf16_to_f32(wd).astype(np.float64)).T
    assert (np.abs(y - ref) <= bound * (1 + 1e-12) + 1e-12).all()
    assert np.abs(y - ref).max() > 0  # h quantisation is visible
