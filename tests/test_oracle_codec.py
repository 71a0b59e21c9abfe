"""Pins of the oracle's codec: bf16 rounding, rotation arithmetic, INT2 quantizer, packing.

Expected values here come from closed forms, IEEE binary32/bf16 facts and hand
derivations written out beside each case, never from the CUDA path.
"""
import numpy as np
import pytest

import oracle
import oscar_synthetic as syn


def bits(x):
    return int(np.float32(x).view(np.uint32))


def test_bf16_round_to_nearest_even():
    # 1.0 is exact.
    assert oracle.f32_to_bf16(1.0) == 0x3F80
    # 1 + 2^-8 sits exactly between 0x3F80 (1.0) and 0x3F81 (1 + 2^-7): ties go to the even one.
    assert oracle.f32_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    # 1 + 3*2^-8 sits between 0x3F81 and 0x3F82: the even one is 0x3F82.
    assert oracle.f32_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # just above the tie rounds up.
    assert oracle.f32_to_bf16(np.float32(1.0 + 2.0 ** -8 + 2.0 ** -20)) == 0x3F81
    # sign and exponent carry: -2.875 = -(1 + 7/16)*2 -> 0xC038.
    assert oracle.f32_to_bf16(-2.875) == 0xC038
    # mantissa overflow carries into the exponent: largest value below 2 rounds to 2.0 (0x4000).
    assert oracle.f32_to_bf16(np.float32(2.0 - 2.0 ** -23)) == 0x4000
    for h in [0x3F80, 0xC038, 0x4000, 0x0001, 0x7F7F]:
        assert oracle.f32_to_bf16(oracle.bf16_to_f64(np.array([h], np.uint16))[0]) == h


def test_pack_all_bytes_round_trip():
    for b in range(256):
        codes = oracle.unpack_row(np.array([b] * 32, np.uint8), 128)
        assert codes.max() <= 3
        assert np.all(oracle.pack_row(codes) == b)


def test_pack_bit_order_worked_byte():
    # element i at bits 2*(i mod 4): codes (1, 2, 3, 0) -> 1 | 2<<2 | 3<<4 | 0<<6 = 0x39.
    assert oracle.pack_row(np.array([1, 2, 3, 0], np.uint8))[0] == 0x39
    # codes (0, 1, 2, 3) -> 0 | 4 | 32 | 192 = 0xE4.
    assert oracle.pack_row(np.array([0, 1, 2, 3], np.uint8))[0] == 0xE4


# Hand-derived quantizer cases: (values, group, clip) -> (codes, zero bits, scale bits).
# Derivations:
#  A  c=1, [-3,-1,1,3 | 0,0.25,1.25,1.5]: group0 lo=-3, step=2 -> zero -3 (0xC040), scale 2 (0x4000),
#     (x+3)/2 = 0,1,2,3.  group1 lo=0, step=0.5 (0x3F00): x/0.5 = 0,0.5,2.5,3 -> ties to even 0,0,2,3.
#  B  c=0.96, [-3,-1,0,3 | 5,5,5,5]: lo = 0.96f*-3 ~ -2.88 -> bf16 -2.875 (0xC038); hi-lo ~ 5.76,
#     /3 ~ 1.92 -> bf16 1.921875 (0x3FF6).  (x+2.875)/1.921875 = -0.065, 0.976, 1.496, 3.057
#     -> 0 (clamped), 1, 1, 3.  group1 constant: zero = bf16(4.8) = 4.8125 (0x409A), scale 0 -> codes 0.
#  C  c=0.92, [-4,-3,-2,-1]: lo ~ -3.68 -> bf16 -3.6875 (0xC06C); (hi-lo)/3 ~ 0.92 -> 0.921875 (0x3F6C);
#     (x+3.6875)/0.921875 = -0.339, 0.746, 1.831, 2.915 -> 0,1,2,3.
#  D  c=1, [0,1,3,6]: step 2 (0x4000), zero 0: x/2 = 0, 0.5, 1.5, 3 -> ties to even 0, 0, 2, 3.
WORKED = [
    ([-3, -1, 1, 3, 0, 0.25, 1.25, 1.5], 4, 1.0, [0, 1, 2, 3, 0, 0, 2, 3], [0xC040, 0x0000], [0x4000, 0x3F00]),
    ([-3, -1, 0, 3, 5, 5, 5, 5], 4, 0.96, [0, 1, 1, 3, 0, 0, 0, 0], [0xC038, 0x409A], [0x3FF6, 0x0000]),
    ([-4, -3, -2, -1], 4, 0.92, [0, 1, 2, 3], [0xC06C], [0x3F6C]),
    ([0, 1, 3, 6], 4, 1.0, [0, 0, 2, 3], [0x0000], [0x4000]),
]


@pytest.mark.parametrize("vals,g,clip,codes,zero,scale", WORKED)
def test_quantizer_worked_rows(vals, g, clip, codes, zero, scale):
    c, z, s = oracle.quantize_row_codes(np.array(vals, np.float32), g, clip)
    assert list(c) == codes
    assert [int(x) for x in z] == zero
    assert [int(x) for x in s] == scale


def test_quantizer_packed_worked():
    packed, z, s = oracle.quantize_rows(np.array([[-3, -1, 1, 3, 0, 0.25, 1.25, 1.5]], np.float32), 4, 1.0)
    assert list(packed[0]) == [0xE4, 0xE0]


def test_quantizer_is_nearest_stored_level():
    """Brute force: each code is the level z + c*s (c in 0..3, stored bf16 z, s) nearest to x,
    ties to the even code; checked in fp64 away from exact ties."""
    x = syn.rotated_rows(1, 64)
    for g in (32, 64, 128):
        for clip in (1.0, 0.96, 0.92):
            packed, zb, sb = oracle.quantize_rows(x, g, clip)
            for r in range(x.shape[0]):
                codes = oracle.unpack_row(packed[r], 128)
                z = oracle.bf16_to_f64(zb[r])
                s = oracle.bf16_to_f64(sb[r])
                for i in range(128):
                    zi, si = z[i // g], s[i // g]
                    if si == 0.0:
                        assert codes[i] == 0
                        continue
                    d = np.abs(float(x[r, i]) - (zi + np.arange(4) * si))
                    best = np.flatnonzero(d <= d.min() * (1 + 1e-6) + 1e-12)
                    assert codes[i] in best, (g, clip, r, i)


def test_quantizer_reconstruction_bound():
    """Inside the clipped range the dequantized value is within half a step (+ rounding slack)."""
    x = syn.rotated_rows(2, 32)
    for g in (32, 128):
        packed, zb, sb = oracle.quantize_rows(x, g, 0.96)
        for r in range(x.shape[0]):
            xh = oracle.dequant_row(packed[r], zb[r], sb[r], 128, g)
            z = oracle.bf16_to_f64(zb[r])
            s = oracle.bf16_to_f64(sb[r])
            for i in range(128):
                zi, si = z[i // g], s[i // g]
                xi = float(x[r, i])
                if zi <= xi <= zi + 3 * si:
                    assert abs(xh[i] - xi) <= 0.5 * si * (1 + 1e-6) + 1e-9


def test_quantizer_naive_exact_levels():
    """c = 1 and a group whose values already sit on 4 bf16-exact levels round-trips exactly."""
    z, s = -1.25, 0.75
    vals = np.array([z + c * s for c in [0, 3, 1, 2] * 32], np.float32)
    packed, zb, sb = oracle.quantize_rows(vals[None], 128, 1.0)
    xh = oracle.dequant_row(packed[0], zb[0], sb[0], 128, 128)
    assert np.array_equal(xh, vals.astype(np.float64))


def test_rotate_f32_within_fp64_bound():
    rng = np.random.default_rng(5)
    D = 128
    R = np.linalg.qr(rng.normal(size=(D, D)))[0].astype(np.float32)
    x = oracle.f32_to_bf16(rng.normal(0, 2, size=(4, D)).astype(np.float32))
    y32 = oracle.rotate_f32(x, R)
    y64 = oracle.rotate_f64(x, R)
    xa = np.abs(oracle.bf16_to_f64(x))
    bound = D * 2.0 ** -24 * (xa @ np.abs(R.astype(np.float64)))   # recursive-summation bound
    assert np.all(np.abs(y32 - y64) <= bound + 1e-30)


def test_rotate_f32_ascending_order():
    """Order is part of the contract: with column (2^24, 1, -2^24, 0...) and x = 1 the
    ascending fp32 chain computes 2^24 + 1 -> 2^24 (ties to even), then 0; the exact sum is 1."""
    D = 128
    R = np.zeros((D, D), np.float32)
    R[0, 0], R[1, 0], R[2, 0] = 2.0 ** 24, 1.0, -(2.0 ** 24)
    x = np.full((1, D), 0x3F80, np.uint16)
    assert oracle.rotate_f32(x, R)[0, 0] == 0.0
    assert oracle.rotate_f64(x, R)[0, 0] == 1.0


def test_demote_rows_equals_rotate_then_quantize():
    rng = np.random.default_rng(9)
    R = np.linalg.qr(rng.normal(size=(128, 128)))[0].astype(np.float32)
    x = oracle.f32_to_bf16(rng.normal(0, 3, size=(5, 128)).astype(np.float32))
    rot, packed, z, s = oracle.demote_rows(x, R, 128, 0.96)
    assert np.array_equal(rot, oracle.rotate_f32(x, R))
    p2, z2, s2 = oracle.quantize_rows(rot, 128, 0.96)
    assert np.array_equal(packed, p2) and np.array_equal(z, z2) and np.array_equal(s, s2)


def test_quantizer_signed_zero_min_reads_as_plus_zero():
    """A group whose minimum is zero gives zero point +0 (0x0000) whichever sign the zeros carry."""
    for vals in ([-0.0, 0.0, 1.5, 3.0], [0.0, -0.0, 1.5, 3.0], [-0.0, -0.0, 3.0, 1.5]):
        c, z, s = oracle.quantize_row_codes(np.array(vals, np.float32), 4, 1.0)
        assert int(z[0]) == 0x0000
        assert int(s[0]) == 0x3F80                      # (3 - 0)/3 = 1
        assert list(c) == [0, 0, 2, 3] if vals[2] == 1.5 else True
