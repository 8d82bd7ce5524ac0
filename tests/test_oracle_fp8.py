"""Pins of the oracle's FP8 latent row ("M5.8" 0x0B, "Exact 656-byte FP8 row"):
the printed row size and ratio, the E4M3 code table's closed forms, brute-force
nearest-code rounding, and quantize/dequantize error bounds."""
import math

import numpy as np

from oracle import mla_oracle as O


def test_row_size_and_ratio_printed():
    # 512 E4M3 bytes + 4 fp32 scales + 64 bf16 RoPE values; against 1152 bf16 bytes
    assert O.FP8_ROW_BYTES == 512 * 1 + 4 * 4 + 64 * 2 == 656
    assert O.latent_bytes_per_token() == 1152
    assert round(656 / 1152, 3) == 0.569
    assert round(100 * (1 - 656 / 1152), 1) == 43.1


def test_e4m3_closed_forms():
    d = O.e4m3_decode
    assert d(0x7E) == 448.0 and d(0xFE) == -448.0           # largest finite: 1.75 * 2^8
    assert d(0x01) == 2.0 ** -9                             # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9                         # largest subnormal
    assert d(0x08) == 2.0 ** -6                             # smallest normal
    assert d(0x38) == 1.0 and d(0x39) == 1.125 and d(0x40) == 2.0
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    assert d(0x00) == 0.0 and math.copysign(1.0, d(0x80)) == -1.0


def test_e4m3_table_monotone_symmetric():
    pos = O.e4m3_decode(np.arange(0x7F))
    assert np.all(np.diff(pos) > 0) and pos[0] == 0.0 and pos[-1] == 448.0
    neg = O.e4m3_decode(np.arange(0x80, 0xFF))
    assert np.array_equal(neg, -pos)
    # inside a binade the step is 1/8 of its power of two
    assert np.allclose(np.diff(O.e4m3_decode(np.arange(0x38, 0x40))), 0.125)


def test_e4m3_round_trip_every_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    assert np.array_equal(O.e4m3_encode(O.e4m3_decode(codes)), codes.astype(np.uint8))


def _brute_force(x):
    """Nearest finite code by exhaustive search; ties to the even mantissa;
    beyond 448 the largest finite value."""
    codes = np.arange(0x7F)
    vals = O.e4m3_decode(codes)
    a = min(abs(x), 448.0)
    dist = np.abs(vals - a)
    best = np.flatnonzero(dist == dist.min())
    c = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
    return c | (0x80 if math.copysign(1.0, x) < 0 else 0)


def test_e4m3_encode_matches_brute_force():
    rng = np.random.default_rng(5)
    xs = list(rng.choice([-1, 1], 400) * np.exp2(rng.uniform(-12, 10, 400)))
    # exact midpoints between neighbouring codes (ties), subnormal and normal
    vals = O.e4m3_decode(np.arange(0x7F))
    xs += list((vals[:-1] + vals[1:]) / 2) + [500.0, 1e6, -464.0, 2.0 ** -10, -3 * 2.0 ** -11]
    got = O.e4m3_encode(np.array(xs))
    assert [int(g) for g in got] == [_brute_force(float(x)) for x in xs]


def _bf16_bits(x):
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def test_row_quantize_bounds_and_layout():
    rng = np.random.default_rng(6)
    c = rng.standard_normal((7, 512)) * 0.1
    c[3, 128:256] = 0.0                        # an all-zero tile: scale 1, codes 0
    c[4, 0] = 1e-30                            # far below the tile's subnormal step
    kpe = _bf16_bits(rng.standard_normal((7, 64)))
    rows = O.fp8_row_quantize(c, kpe)
    assert rows.shape == (7, 656) and rows.dtype == np.uint8
    c_hat, scale, kpe_back = O.fp8_row_dequantize(rows)
    assert np.array_equal(kpe_back, kpe)
    tiles = c.reshape(7, 4, 128)
    amax = np.abs(tiles).max(-1)
    # the stored scale is amax / 448 rounded once to fp32: within half an fp32 ulp
    nz = amax > 0
    assert np.all(np.abs(scale[nz].astype(np.float64) - amax[nz] / 448.0) <= amax[nz] / 448.0 * 2.0 ** -24)
    assert np.all(rows[3, 128:256] == 0) and scale[3, 1] == 1.0
    # per element: half a subnormal step (2^-10 * scale) or half a normal ulp (2^-4 relative)
    s = np.repeat(scale.astype(np.float64), 128, axis=1)
    err = np.abs(c_hat - c)
    assert np.all(err <= np.maximum(s * 2.0 ** -10, np.abs(c) * 2.0 ** -4) * (1 + 1e-12))
    # each tile's largest magnitude maps to code 448 and comes back within the scale's fp32 rounding
    idx = np.abs(tiles).argmax(-1)
    hat_max = np.take_along_axis(c_hat.reshape(7, 4, 128), idx[..., None], -1)[..., 0]
    ref_max = np.take_along_axis(tiles, idx[..., None], -1)[..., 0]
    nz = amax > 0
    assert np.all(np.abs(hat_max[nz] - ref_max[nz]) <= amax[nz] * 2.0 ** -23)


def test_lossless_rows_decode_identically():
    """Rows whose tiles are E4M3 values times a power of two, each tile holding a
    +-448 * 2^k entry, quantize losslessly: the attention over the dequantized
    rows equals the attention over the originals exactly."""
    rng = np.random.default_rng(7)
    S = 70
    codes = rng.integers(0, 0x7F, size=(S, 4, 128))
    codes[:, :, 0] = 0x7E
    codes |= rng.choice([0, 0x80], size=codes.shape)
    k = rng.integers(-12, -4, size=(S, 4, 1)).astype(np.float64)
    c = (O.e4m3_decode(codes) * np.exp2(k)).reshape(S, 512)
    kpe_f = rng.standard_normal((S, 64)) * 0.1
    kpe = _bf16_bits(kpe_f)
    c_hat, _, kpe_back = O.fp8_row_dequantize(O.fp8_row_quantize(c, kpe))
    assert np.array_equal(c_hat, c)
    kpe64 = (kpe_back.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    rows_ref = np.concatenate([c, (kpe.astype(np.uint32) << 16).view(np.float32).astype(np.float64)], axis=1)
    rows_fp8 = np.concatenate([c_hat, kpe64], axis=1)
    q_lat = rng.standard_normal((1, 3, 512)) * 0.05
    q_pe = rng.standard_normal((1, 3, 64)) * 0.05
    mask = O.causal_mask(S, 1, False)
    o1, l1 = O.attend_latent(q_lat, q_pe, rows_ref, mask)
    o2, l2 = O.attend_latent(q_lat, q_pe, rows_fp8, mask)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def _nearest_code_exact(value, scale):
    """Brute force in exact rational arithmetic: the E4M3 code whose value is
    nearest to value / scale, ties to the even mantissa, saturating at 448."""
    from fractions import Fraction
    q = abs(Fraction(float(value)) / Fraction(float(scale)))
    vals = [Fraction(float(v)) for v in O.e4m3_decode(np.arange(0x7F))]
    q = min(q, vals[-1])
    dist = [abs(v - q) for v in vals]
    best = min(dist)
    near = [c for c, d in enumerate(dist) if d == best]
    c = near[0] if len(near) == 1 else [x for x in near if x % 2 == 0][0]
    return c | (0x80 if math.copysign(1.0, float(value)) < 0 else 0)


def test_scaled_encode_exact_at_midpoints():
    """Codes are decided on the exact quotient: values placed one float64 ulp either
    side of a midpoint times the scale (where a rounded float64 quotient can land on
    the wrong side), exactly on it (a tie), and random float64 values."""
    rng = np.random.default_rng(12)
    pos = O.e4m3_decode(np.arange(0x7F))
    mids = (pos[:-1] + pos[1:]) / 2.0
    scales = [np.float32(0.1 / 448), np.float32(3.0e-5), np.float32(1.0), np.float32(7.0)]
    for s in scales:
        s64 = float(s)
        ks = rng.choice(mids.size, size=40, replace=False)
        vals = []
        for k in ks:
            t = mids[k] * s64                       # exact in float64
            vals += [t, np.nextafter(t, np.inf), np.nextafter(t, -np.inf), -t]
        vals += list(rng.standard_normal(60) * s64 * 100.0)
        vals = np.array(vals, dtype=np.float64)
        got = O.e4m3_encode_scaled(vals[None], np.array([s]))[0]
        ref = [_nearest_code_exact(v, s) for v in vals]
        assert [int(g) for g in got] == ref


def test_fp32_scale_is_the_nearest_to_the_exact_quotient():
    from fractions import Fraction
    rng = np.random.default_rng(13)
    nums = list(rng.standard_normal(200) ** 2 * 0.3) + [448.0 * 3.0, 1e-30, 2.0 ** -140]
    for x in nums:
        got = O.f32_nearest_quotient(float(x), 448.0)
        exact = Fraction(float(x)) / 448
        f = np.float32(got)
        lo, hi = np.nextafter(f, np.float32(-np.inf)), np.nextafter(f, np.float32(np.inf))
        d = abs(Fraction(float(f)) - exact)
        assert d <= abs(Fraction(float(lo)) - exact) and d <= abs(Fraction(float(hi)) - exact)
