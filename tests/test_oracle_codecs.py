"""Pins for the oracle's element codecs.

Each check comes from outside the oracle's own code: the spec tables in
tests/golden/format_tables.txt, torch's float8 casts (a library routine), an
exact-rational brute-force search over all codes, and binary32 facts read off
Python's own float decomposition.
"""
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "format_tables.txt")


def f32(x: float) -> float:
    return struct.unpack("<f", struct.pack("<f", x))[0]


def f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def bits_f32(u: int) -> float:
    return struct.unpack("<f", struct.pack("<I", u & 0xFFFFFFFF))[0]


def _golden():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        fmt, code, val = line.split()
        rows.append((fmt, int(code, 16), float(val)))
    return rows


def _same(a, b):
    if math.isnan(b):
        return math.isnan(a)
    return a == b and math.copysign(1, a) == math.copysign(1, b)


def test_golden_spec_tables(orc):
    dec = {"e4m3": orc.dec_e4m3, "e2m1": orc.dec_e2m1, "e8m0": orc.dec_e8m0}
    for fmt, code, val in _golden():
        assert _same(dec[fmt](code), val), (fmt, hex(code))


def test_e4m3_decode_matches_torch_all_codes(orc):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).tolist()
    for c in range(256):
        assert _same(orc.dec_e4m3(c), ref[c]), hex(c)


def test_e8m0_decode_matches_torch(orc):
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("torch without float8_e8m0fnu")
    codes = torch.arange(255, dtype=torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).tolist()
    for c in range(255):
        assert orc.dec_e8m0(c) == ref[c] == 2.0 ** (c - 127), c


def _finite_e4m3(orc):
    return [(c, orc.dec_e4m3(c)) for c in range(256) if not math.isnan(orc.dec_e4m3(c))]


def _finite_e2m1(orc):
    return [(c, orc.dec_e2m1(c)) for c in range(16)]


def brute_nearest(v: float, table, maxval: float, mant_bits: int) -> int:
    """Nearest code by exact rational distance; ties go to the code whose
    mantissa LSB is 0; magnitudes beyond maxval saturate; the sign of v is kept.
    ``mant_bits`` documents the format; the code LSB is the mantissa LSB in both."""
    neg = math.copysign(1.0, v) < 0
    a = Fraction(abs(v))
    if a > Fraction(maxval):
        a = Fraction(maxval)
    best, bestd = None, None
    for c, val in table:
        if (math.copysign(1.0, val) < 0) != neg:
            continue
        d = abs(Fraction(abs(val)) - a)
        if bestd is None or d < bestd:
            best, bestd = [c], d
        elif d == bestd:
            best.append(c)
    if len(best) == 1:
        return best[0]
    even = [c for c in best if c & 1 == 0]      # the code LSB is the mantissa LSB
    assert len(even) == 1, (v, best)
    return even[0]


def test_e4m3_roundtrip_every_finite_code(orc):
    for c, val in _finite_e4m3(orc):
        assert orc.enc_e4m3(val) == c, hex(c)


def test_e4m3_midpoints_tie_to_even_and_neighbours(orc):
    table = _finite_e4m3(orc)
    pos = sorted({abs(v) for _, v in table})
    for lo, hi in zip(pos[:-1], pos[1:]):
        mid = (lo + hi) / 2                       # exact in binary32 here
        assert f32(mid) == mid
        for sgn in (1.0, -1.0):
            v = sgn * mid
            assert orc.enc_e4m3(v) == brute_nearest(v, table, 448.0, 3), v
            below = bits_f32(f32_bits(mid) - 1) * sgn
            above = bits_f32(f32_bits(mid) + 1) * sgn
            assert orc.dec_e4m3(orc.enc_e4m3(below)) == sgn * lo
            assert orc.dec_e4m3(orc.enc_e4m3(above)) == sgn * hi


def test_e4m3_random_vs_bruteforce_and_torch(orc):
    rng = np.random.default_rng(7)
    table = _finite_e4m3(orc)
    vals = np.concatenate([
        rng.standard_normal(400) * 100, rng.standard_normal(300) * 1e-2,
        rng.standard_normal(200) * 1e-3, rng.uniform(440, 600, 50) * rng.choice([-1, 1], 50),
        np.ldexp(rng.uniform(1, 2, 50), rng.integers(-14, -8, 50)),
    ]).astype(np.float32)
    ours = [orc.enc_e4m3(float(v)) for v in vals]
    for v, c in zip(vals.tolist(), ours):
        assert c == brute_nearest(v, table, 448.0, 3), v
    in_range = np.abs(vals) <= 448
    t = torch.from_numpy(vals[in_range]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(t, np.array(ours, np.uint8)[in_range])


def test_e4m3_saturation_and_signed_zero(orc):
    for v in (448.0, 449.0, 464.0, 480.0, 1e6, 3.0e38):
        assert orc.enc_e4m3(v) == 0x7E
        assert orc.enc_e4m3(-v) == 0xFE
    assert orc.enc_e4m3(0.0) == 0x00
    assert orc.enc_e4m3(-0.0) == 0x80
    assert orc.enc_e4m3(-2.0 ** -11) == 0x80       # rounds to zero, sign kept
    assert orc.enc_e4m3(2.0 ** -10) == 0x00        # exactly half the min subnormal: tie to even 0
    assert orc.enc_e4m3(3 * 2.0 ** -10) == 0x02    # 1.5 min subnormals -> even code 2
    assert orc.enc_e4m3(3 * 2.0 ** -11) == 0x01    # 0.75 min subnormals -> code 1


def test_e2m1_every_value_roundtrip_and_ties(orc):
    table = _finite_e2m1(orc)
    for c, val in table:
        assert orc.enc_e2m1(val) == c or (val == 0 and orc.enc_e2m1(val) in (0, 8))
    expect = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0, 7.0: 6.0, 100.0: 6.0}
    for v, want in expect.items():
        assert orc.dec_e2m1(orc.enc_e2m1(v)) == want, v
        assert orc.dec_e2m1(orc.enc_e2m1(-v)) == -want, v


def test_e2m1_random_vs_bruteforce(orc):
    rng = np.random.default_rng(11)
    table = _finite_e2m1(orc)
    vals = np.concatenate([rng.uniform(-7, 7, 2000), rng.uniform(-1, 1, 500)]).astype(np.float32)
    for v in vals.tolist():
        assert orc.enc_e2m1(v) == brute_nearest(v, table, 6.0, 1), v


def test_bf16_rne_matches_torch(orc):
    rng = np.random.default_rng(3)
    u = rng.integers(0, 2**32, 20000, dtype=np.uint64).astype(np.uint32)
    u = u[(u & 0x7F800000) != 0x7F800000]                # finite only
    ties = (rng.integers(0, 2**15, 2000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    u = np.concatenate([u, ties, ties | 0x10000]).astype(np.uint32)
    f = u.view(np.float32)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ref_fin = np.isfinite(torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())
    ours = np.array([orc.f32_to_bf16(float(x)) for x in f], np.uint16)
    assert np.array_equal(ours[ref_fin], ref[ref_fin])


def test_floor_log2_vs_frexp(orc):
    rng = np.random.default_rng(5)
    vals = np.concatenate([np.abs(rng.standard_normal(3000)) * 10.0 ** rng.integers(-30, 30, 3000),
                           np.array([2.0 ** -149, 2.0 ** -140, 2.0 ** -126, 1.0, 2.0, 3.0, 2.0 ** 127])])
    vals = vals.astype(np.float32)
    for v in vals.tolist():
        if v == 0:
            continue
        m, e = math.frexp(v)                     # v = m * 2^e, 0.5 <= m < 1
        assert orc.floor_log2(v) == e - 1, v
