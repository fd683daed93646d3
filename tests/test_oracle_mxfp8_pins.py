"""Pins of the oracle's MXFP8 activation format (the lossy variant).

Kimi K3 is trained quantisation-aware with MXFP8 activations (Deltafin
analysis, section 2.1); the variant rounds the routed experts' inputs to that
format. The element type is FP8 E4M3 and the block an OCP microscaling block
of 32 with an E8M0 exponent. Each check below is independent of the oracle's
own code: ml_dtypes' float8_e4m3fn (a library cast, ties to even), a decoder
written here from the format's fields, hand-worked ties and closed forms for
the block exponent. A slip in the bias, the subnormal spacing, the tie rule,
the saturation, the block exponent (off by one in floor(log2)) or the block
index fails at least one of them. No CUDA here.
"""
import math

import numpy as np
import pytest

import oracle as orc


def e4m3_from_fields(code):
    """OCP E4M3: sign bit 7, 4-bit exponent (bias 7), 3-bit mantissa;
    exponent 0 is subnormal (2^-6 * m/8); S.1111.111 is NaN, no inf."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 15
    m = code & 7
    if e == 15 and m == 7:
        return math.nan
    if e == 0:
        return s * m / 8.0 * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def test_e4m3_table_against_fields():
    for c in range(256):
        a, b = orc.e4m3_value(c), e4m3_from_fields(c)
        assert (math.isnan(a) and math.isnan(b)) or a == b, c
    assert orc.e4m3_value(0x7E) == 448.0          # largest finite
    assert orc.e4m3_value(0x01) == 2.0 ** -9      # smallest subnormal
    assert orc.e4m3_value(0x08) == 2.0 ** -6      # smallest normal
    assert orc.e4m3_value(0x38) == 1.0


def test_e4m3_table_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    ref = np.arange(256, dtype=np.uint8).view(ml.float8_e4m3fn).astype(np.float64)
    got = np.array([orc.e4m3_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(got[ok]))


def test_e4m3_rounding_hand_worked():
    cases = [  # (value, code); a list, since -0.0 == 0.0 as dict keys
        (1.0, 0x38), (1.0625, 0x38),   # halfway 1 .. 1.125: ties to even (1.0)
        (1.1875, 0x3A),                # halfway 1.125 .. 1.25: even is 1.25
        (1.0626, 0x39),
        (2.0 ** -10, 0x00),            # halfway 0 .. 2^-9: ties to 0
        (3 * 2.0 ** -10, 0x02),        # halfway 2^-9 .. 2^-8: even is 2^-8
        (2.0 ** -6, 0x08),
        (15 * 2.0 ** -10, 0x08),       # halfway 7*2^-9 .. 2^-6: even is 2^-6
        (448.0, 0x7E), (460.0, 0x7E), (464.0, 0x7E), (500.0, 0x7E), (1e30, 0x7E),
        (-1000.0, 0xFE), (-0.0, 0x80), (0.0, 0x00),
        (240.0, 0x77), (248.0, 0x78),  # 240 is 1.875*2^7; 248 halfway, even is 256
    ]
    for v, c in cases:
        assert orc.e4m3_from_f64(v) == c, (v, hex(orc.e4m3_from_f64(v)), hex(c))


def test_e4m3_rounding_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(7)
    mag = np.ldexp(rng.uniform(1.0, 2.0, 20000), rng.integers(-14, 10, 20000))
    v = mag * rng.choice([-1.0, 1.0], 20000)
    # every midpoint between neighbouring finite codes, both signs
    vals = np.array([orc.e4m3_value(c) for c in range(0x7F)])
    mids = (vals[:-1] + vals[1:]) / 2
    v = np.concatenate([v, mids, -mids, vals, -vals])
    ref = np.clip(v, -448.0, 448.0).astype(ml.float8_e4m3fn).view(np.uint8)
    got = np.array([orc.e4m3_from_f64(x) for x in v], dtype=np.uint8)
    assert np.array_equal(got, ref)


def independent_block(v):
    """Block exponent from frexp, elements by the ml_dtypes cast."""
    ml = pytest.importorskip("ml_dtypes")
    amax = np.max(np.abs(v))
    if amax == 0:
        sh = -127
    else:
        sh = int(np.frexp(amax)[1]) - 1 - 8
        sh = min(127, max(-127, sh))
    q = np.clip(np.ldexp(v, -sh), -448.0, 448.0).astype(ml.float8_e4m3fn).view(np.uint8)
    return q, sh + 127


def test_block_exponent_closed_form():
    for e in (-20, -7, 0, 1, 5, 40):
        for frac in (1.0, 1.5, 1.999):
            v = np.zeros(32)
            v[3] = -frac * 2.0 ** e   # the largest magnitude, negative
            v[10] = 0.25 * 2.0 ** e
            codes, scales = orc.mxfp8_quantize(v[None, :])
            assert scales[0, 0] == e - 8 + 127
            # the largest element lands in [256, 512) before rounding:
            # 256 and 384 are codes, 511.7 saturates to 448
            want = {1.0: 256.0, 1.5: 384.0, 1.999: 448.0}[frac]
            assert orc.e4m3_value(int(codes[0, 3])) == -want
            assert orc.e4m3_value(int(codes[0, 10])) == 64.0
    # an all-zero block: exponent code 0, zero codes
    codes, scales = orc.mxfp8_quantize(np.zeros((1, 32)))
    assert scales[0, 0] == 0 and not codes.any()
    # clamping at both ends of E8M0
    codes, scales = orc.mxfp8_quantize(np.full((1, 32), 2.0 ** -140))
    assert scales[0, 0] == 0            # 2^-127: the exponent is clamped ...
    assert not codes.any()              # ... and 2^-13 is below half of 2^-9
    codes, scales = orc.mxfp8_quantize(np.full((1, 32), 2.0 ** 140))
    assert scales[0, 0] == 254


def test_quantize_matches_independent_blocks():
    rng = np.random.default_rng(11)
    rows, n = 9, 256
    v = rng.standard_normal((rows, n)) * np.ldexp(1.0, rng.integers(-30, 30, (rows, 1)))
    v[2, 32:64] = 0.0                  # a zero block
    v[3, :32] = 2.0 ** 7               # a constant power-of-two block
    v[4, 5] = 1e6                      # one outlier
    codes, scales = orc.mxfp8_quantize(v)
    for r in range(rows):
        for b in range(n // 32):
            q, s = independent_block(v[r, 32 * b:32 * b + 32])
            assert scales[r, b] == s, (r, b)
            assert np.array_equal(codes[r, 32 * b:32 * b + 32], q), (r, b)


def test_block_index_follows_the_row():
    # one large value per block moves only its own block's exponent
    v = np.ones((2, 128))
    v[1, 70] = 1000.0
    _, scales = orc.mxfp8_quantize(v)
    assert list(scales[0]) == [119] * 4
    assert list(scales[1]) == [119, 119, 127 + 9 - 8, 119]


def test_round_trip_error_bound():
    rng = np.random.default_rng(5)
    v = rng.standard_normal((64, 256))
    back = orc.mxfp8_round(v)
    _, scales = orc.mxfp8_quantize(v)
    X = np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=1)
    a = np.abs(v) / X
    normal = (a >= 2.0 ** -6) & (a <= 448.0)
    # three mantissa bits: half an ulp is at most 2^-4 of the magnitude
    assert np.all(np.abs(back - v)[normal] <= 2.0 ** -4 * np.abs(v)[normal])
    sub = a < 2.0 ** -6
    assert np.all(np.abs(back - v)[sub] <= 2.0 ** -10 * X[sub])
    # relative RMS error of a Gaussian block: E4M3 keeps it near 2-3 %
    rel = np.linalg.norm(back - v) / np.linalg.norm(v)
    assert 0.005 < rel < 0.05


def test_dequant_is_code_times_scale():
    codes = np.arange(64, dtype=np.uint8).reshape(1, 64)
    scales = np.array([[127 + 3, 127 - 2]], dtype=np.uint8)
    v = orc.mxfp8_dequant(codes, scales)
    for i in range(64):
        assert v[0, i] == e4m3_from_fields(i) * 2.0 ** (3 if i < 32 else -2)


def independent_round(v):
    """MXFP8 round trip of the rows of v, block by block, from the
    independent block routine above."""
    ml = pytest.importorskip("ml_dtypes")
    v = np.atleast_2d(np.asarray(v, dtype=np.float64))
    out = np.empty_like(v)
    for r in range(v.shape[0]):
        for b in range(v.shape[1] // 32):
            q, s = independent_block(v[r, 32 * b:32 * b + 32])
            out[r, 32 * b:32 * b + 32] = q.view(ml.float8_e4m3fn).astype(np.float64) * \
                2.0 ** (int(s) - 127)
    return out


def test_layer_with_mxfp8_activations_brute_force():
    """Every routed expert takes MXFP8(x) and its down projection MXFP8(h);
    the router and the shared expert see x exactly."""
    import synth
    from test_oracle_pins import (bf16_bits_to_f64, dequant_ml_dtypes, shared_numpy,
                                  split_span, tiny_layer)
    L, spans, router, shared = tiny_layer(k=2)
    H, I = 256, 64
    x = np.stack([synth.token(0, 0, t, H) for t in range(3)])
    res = np.stack([synth.token(0, 0, t, H, kind=synth.gen.KIND_RESIDUAL) for t in range(3)])
    r = orc.moe_layer_mxfp8(L, x, residual=res)
    exact = orc.moe_layer(L, x, residual=res)
    assert np.array_equal(r["ids"], exact["ids"])
    for t in range(3):
        xd = bf16_bits_to_f64(x[t])
        xq = independent_round(xd)[0]
        logits = router.astype(np.float64) @ xd
        best = sorted(range(8), key=lambda e: (-logits[e], e))[:2]
        w = np.exp(logits[best] - logits[best].max()); w /= w.sum()
        y = np.zeros(H)
        for j, e in enumerate(best):
            gq, gs, uq, us, dq, ds = split_span(spans[e], H, I)
            gx = dequant_ml_dtypes(gq, gs) @ xq
            ux = dequant_ml_dtypes(uq, us) @ xq
            h = gx / (1.0 + np.exp(-gx)) * ux
            assert np.allclose(r["h"][t * 2 + j], h, rtol=1e-12, atol=1e-12 * np.abs(h).max())
            y += w[j] * (dequant_ml_dtypes(dq, ds) @ independent_round(h)[0])
        sh = shared_numpy(*shared[0], xd)
        assert np.allclose(r["routed"][t], y, rtol=1e-10, atol=1e-10 * np.abs(y).max())
        assert np.allclose(r["shared"][t], sh, rtol=1e-12, atol=1e-12)
        assert np.allclose(r["out"][t], y + sh + bf16_bits_to_f64(res[t]), rtol=1e-10,
                           atol=1e-10 * np.abs(y).max())
        # lossy, but only by the format's few per cent
        d = np.linalg.norm(r["routed"][t] - exact["routed"][t]) / np.linalg.norm(exact["routed"][t])
        assert 1e-4 < d < 0.1
    # h_in: the rounding of h decides on the caller's values
    r2 = orc.moe_layer_mxfp8(L, x, residual=res, h_in=r["h"])
    assert np.array_equal(r2["out"], r["out"])
    r3 = orc.moe_layer_mxfp8(L, x, residual=res, h_in=r["h"] * 2.0)
    assert np.allclose(r3["routed"], 2.0 * r["routed"], rtol=1e-12, atol=1e-14)
