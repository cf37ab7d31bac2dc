"""Pins for the oracle's quantizers and dequantizers.

The pages print no worked example for any of these formats, so each quantizer
is pinned by what the formats and the mathematics fix: the amax element lands
on the format maximum, codes are the nearest representable values of x/s
(checked against an exact-rational search over all codes), powers of two
scale through exactly, granules are independent, the packing layout is read
back with an unpacker written from the format description, and
dequant(quant(x)) stays within half a code step of x.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from serving_amax_reduce_gb300 import inputs


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def vals(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


E4M3_POS = None


def e4m3_grid(orc):
    global E4M3_POS
    if E4M3_POS is None:
        E4M3_POS = np.array(sorted({abs(orc.dec_e4m3(c)) for c in range(256)
                                    if not math.isnan(orc.dec_e4m3(c))}))
    return E4M3_POS


E2M1_POS = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)


def half_step(grid: np.ndarray, a: np.ndarray) -> np.ndarray:
    """Half the distance between the two grid points around |a| (saturating)."""
    a = np.minimum(np.abs(a), grid[-1])
    i = np.clip(np.searchsorted(grid, a, side="right"), 1, len(grid) - 1)
    return (grid[i] - grid[i - 1]) / 2


def assert_nearest(dec_codes, target, grid, slack=1e-6):
    """Each decoded code is within half a step of the (unsaturated) target."""
    err = np.abs(dec_codes - np.clip(target, -grid[-1], grid[-1]))
    bound = half_step(grid, target) * (1 + slack) + 1e-300
    bad = err > bound
    assert not bad.any(), (np.argwhere(bad)[:5], dec_codes[bad][:5], target[bad][:5])


def dec_vec(fn, codes):
    lut = np.array([fn(c) for c in range(256)], np.float64)
    return lut[codes]


def rand_bits(shape, seed, std=1.0):
    return bf16_bits(inputs.normal_bf16(shape, std, seed))


# ------------------------------------------------------------------ FP8 scaled
@pytest.mark.parametrize("kind", ["tensor", "token", "block128"])
def test_fp8_amax_maps_to_448_and_codes_are_nearest(orc, kind):
    R, K = 256, 384
    x = bf16_bits(inputs.outlier_channel_bf16(R, K, 77))
    xv = vals(x)
    q = {"tensor": orc.quant_fp8_tensor, "token": orc.quant_fp8_token,
         "block128": orc.quant_fp8_block128}[kind]
    codes, s = q(x)
    if kind == "tensor":
        s_full = np.full((R, K), float(s))
        gran = [(slice(0, R), slice(0, K))]
    elif kind == "token":
        s_full = np.repeat(np.asarray(s, np.float64)[:, None], K, 1)
        gran = [(slice(i, i + 1), slice(0, K)) for i in range(R)]
    else:
        s_full = np.kron(np.asarray(s, np.float64), np.ones((128, 128)))
        gran = [(slice(i, i + 128), slice(j, j + 128)) for i in range(0, R, 128) for j in range(0, K, 128)]
    d = dec_vec(orc.dec_e4m3, codes)
    for g in gran:
        a = np.abs(xv[g]).max()
        sg = s_full[g].flat[0]
        assert abs(sg * 448 - a) <= a * 2.0 ** -22            # s = amax/448 to binary32 rounding
        at = np.abs(xv[g]) == a
        assert np.all(np.abs(d[g][at]) == 448.0)
    assert_nearest(d, xv / s_full, e4m3_grid(orc), slack=1e-5)


@pytest.mark.parametrize("kind", ["tensor", "token", "block128"])
def test_fp8_sign_symmetry_power_of_two_and_zero(orc, kind):
    q = {"tensor": orc.quant_fp8_tensor, "token": orc.quant_fp8_token,
         "block128": orc.quant_fp8_block128}[kind]
    t = inputs.normal_bf16((128, 256), 0.02, 5)
    c1, s1 = q(bf16_bits(t))
    c2, s2 = q(bf16_bits(-t))
    assert np.array_equal(c2, c1 ^ 0x80) and np.array_equal(s1, s2)
    c3, s3 = q(bf16_bits(t * 4))
    assert np.array_equal(c3, c1) and np.array_equal(np.asarray(s3), np.asarray(s1) * 4)
    cz, sz = q(np.zeros((128, 256), np.uint16))
    assert not cz.any() and np.all(np.asarray(sz) == 1.0)


def test_fp8_block_granules_are_independent(orc):
    w = rand_bits((256, 384), 9, 0.02)
    c1, s1 = orc.quant_fp8_block128(w)
    w2 = w.copy()
    w2[128:256, 256:384] = bf16_bits(inputs.normal_bf16((128, 128), 50.0, 10))
    c2, s2 = orc.quant_fp8_block128(w2)
    changed = np.zeros((2, 3), bool)
    changed[1, 2] = True
    assert np.array_equal(s1[~changed], s2[~changed]) and s1[1, 2] != s2[1, 2]
    mask = np.ones((256, 384), bool)
    mask[128:, 256:] = False
    assert np.array_equal(c1[mask], c2[mask])


def test_fp8_codes_follow_the_reciprocal_form(orc):
    """Reading R1: code = E4M3(x * fl(448 / amax)), not E4M3(x / fl(amax / 448)).
    On constructed rows where the two differ, every FP8 granule kind (token,
    1 x 128 group, tensor) gives the reciprocal form's code, found by an
    exact-rational search over all E4M3 codes."""
    from hard_cases import fp8_reciprocal_candidates, rows_of_pairs
    from test_oracle_codecs import brute_nearest
    table = [(c, orc.dec_e4m3(c)) for c in range(256) if not math.isnan(orc.dec_e4m3(c))]
    f32 = np.float32
    pairs, want = [], []
    for a, x in fp8_reciprocal_candidates([v for _, v in table]):
        c_mul = brute_nearest(float(f32(x) * (f32(448) / f32(a))), table, 448.0, 3)
        c_div = brute_nearest(float(f32(x) / (f32(a) / f32(448))), table, 448.0, 3)
        if c_mul != c_div:
            pairs.append((a, x))
            want.append(c_mul)
    assert len(pairs) >= 100                       # the readings really differ on these rows
    rows = rows_of_pairs(pairs, 128)
    codes, scales = orc.quant_fp8_token(rows)
    assert list(codes[:, 1]) == want
    assert np.array_equal(scales, np.array([f32(a) / f32(448) for a, _ in pairs], np.float32))
    gcodes, _ = orc.quant_fp8_group128(rows)
    assert list(gcodes[:, 1]) == want
    for (a, x), w, row in list(zip(pairs, want, rows))[:20]:
        tcodes, _ = orc.quant_fp8_tensor(row[None, :])
        assert tcodes[0, 1] == w
    from hard_cases import tiles_of_pairs
    stride = len(pairs) // 64
    tiles = tiles_of_pairs(pairs[::stride])
    bcodes, _ = orc.quant_fp8_block128(tiles)
    assert list(bcodes[0, 1::128]) == want[::stride][:64]


def test_fp8_group128_amax_maps_to_448_and_codes_are_nearest(orc):
    R, K = 64, 512
    x = bf16_bits(inputs.outlier_channel_bf16(R, K, 81))
    xv = vals(x)
    codes, s = orc.quant_fp8_group128(x)
    assert s.shape == (R, K // 128)
    s_full = np.repeat(np.asarray(s, np.float64), 128, 1)
    d = dec_vec(orc.dec_e4m3, codes)
    for i in range(R):
        for g in range(K // 128):
            blk = np.abs(xv[i, g * 128:(g + 1) * 128])
            a = blk.max()
            assert abs(s[i, g] * 448 - a) <= a * 2.0 ** -22    # s = amax/448 to binary32 rounding
            assert np.all(np.abs(d[i, g * 128:(g + 1) * 128][blk == a]) == 448.0)
    assert_nearest(d, xv / s_full, e4m3_grid(orc), slack=1e-5)


def test_fp8_group128_reduces_to_token_when_k_is_128(orc):
    # with K = 128 a row is one group: the same codes and scales as per-token quantization
    x = rand_bits((96, 128), 83)
    c1, s1 = orc.quant_fp8_group128(x)
    c2, s2 = orc.quant_fp8_token(x)
    assert np.array_equal(c1, c2) and np.array_equal(s1[:, 0].view(np.uint32), s2.view(np.uint32))


def test_fp8_group128_groups_are_independent_and_dequant_close(orc):
    x = rand_bits((8, 512), 85)
    c1, s1 = orc.quant_fp8_group128(x)
    x2 = x.copy()
    x2[5, 256:384] = bf16_bits(inputs.normal_bf16((1, 128), 1000.0, 86))[0]
    c2, s2 = orc.quant_fp8_group128(x2)
    changed = np.zeros((8, 4), bool)
    changed[5, 2] = True
    assert np.array_equal(s1[~changed], s2[~changed]) and s1[5, 2] != s2[5, 2]
    keep = np.ones((8, 512), bool)
    keep[5, 256:384] = False
    assert np.array_equal(c1[keep], c2[keep])
    # groups 10^k apart: a transposed scale index would miss by orders of magnitude
    xv = vals(x) * np.repeat(10.0 ** np.arange(4)[None, :], 128, 1)
    xb = bf16_bits(torch.from_numpy(xv).to(torch.bfloat16))
    c, sc = orc.quant_fp8_group128(xb)
    xh = orc.dequant_fp8_group128(c, sc)
    unit = np.repeat(np.asarray(sc, np.float64), 128, 1)
    bound = half_step(e4m3_grid(orc), vals(xb) / unit) * unit * (1 + 1e-5)
    assert np.all(np.abs(xh - vals(xb)) <= bound)


def test_fp8_token_rows_are_independent(orc):
    x = rand_bits((8, 512), 12)
    c1, s1 = orc.quant_fp8_token(x)
    x2 = x.copy()
    x2[3] = bf16_bits(inputs.normal_bf16((1, 512), 100.0, 13))[0]
    c2, s2 = orc.quant_fp8_token(x2)
    keep = np.arange(8) != 3
    assert np.array_equal(c1[keep], c2[keep]) and np.array_equal(s1[keep], s2[keep])


@pytest.mark.parametrize("kind", ["tensor", "token", "block128"])
def test_fp8_dequant_close_and_index_layout(orc, kind):
    """dequant(quant(x)) within half an E4M3 step of x; with granules of very
    different magnitude a transposed scale index would miss by orders of magnitude."""
    R, K = 256, 384
    x = vals(rand_bits((R, K), 21))
    x *= np.kron(10.0 ** np.arange(6).reshape(2, 3), np.ones((128, 128)))
    xb = bf16_bits(torch.from_numpy(x).to(torch.bfloat16))
    xv = vals(xb)
    if kind == "tensor":
        c, s = orc.quant_fp8_tensor(xb)
        xh = orc.dequant_fp8_tensor(c, s)
        sf = float(s)
    elif kind == "token":
        c, s = orc.quant_fp8_token(xb)
        xh = orc.dequant_fp8_token(c, s)
        sf = np.asarray(s, np.float64)[:, None]
    else:
        c, s = orc.quant_fp8_block128(xb)
        xh = orc.dequant_fp8_block128(c, s)
        sf = np.kron(np.asarray(s, np.float64), np.ones((128, 128)))
    err = np.abs(xh - xv)
    bound = half_step(e4m3_grid(orc), xv / sf) * sf * (1 + 1e-5)
    assert np.all(err <= bound)


# ------------------------------------------------------------------ MXFP8
def test_mxfp8_shared_exponent_rule(orc):
    x = bf16_bits(inputs.outlier_channel_bf16(64, 512, 31))
    xv = vals(x)
    codes, sc = orc.quant_mxfp8(x)
    scale = np.vectorize(orc.dec_e8m0)(sc)
    amax = np.abs(xv).reshape(64, 16, 32).max(-1)
    # largest power of two <= amax, divided by 2^8 (the largest E4M3 power of two)
    p2 = np.array([[2.0 ** (math.frexp(a)[1] - 1) for a in row] for row in amax])
    assert np.array_equal(scale, p2 / 256)
    assert np.all(np.log2(scale) == np.round(np.log2(scale)))          # powers of two
    d = dec_vec(orc.dec_e4m3, codes)
    target = xv / np.repeat(scale, 32, 1)                               # exact: power-of-two scaling
    assert_nearest(d, target, e4m3_grid(orc))
    # the amax element lands in [256, 448]
    at = np.abs(xv).reshape(64, 16, 32) == amax[..., None]
    dm = np.abs(d).reshape(64, 16, 32)[at]
    assert np.all((dm >= 256) & (dm <= 448))


def test_mxfp8_exact_bruteforce_small(orc):
    from test_oracle_codecs import brute_nearest
    table = [(c, orc.dec_e4m3(c)) for c in range(256) if not math.isnan(orc.dec_e4m3(c))]
    x = bf16_bits(inputs.normal_bf16((2, 64), 3.0, 41))
    codes, sc = orc.quant_mxfp8(x)
    xv = vals(x)
    for i in range(2):
        for k in range(64):
            v = xv[i, k] / orc.dec_e8m0(int(sc[i, k // 32]))
            assert codes[i, k] == brute_nearest(v, table, 448.0, 3)


def test_mxfp8_scale_by_two_and_zero(orc):
    t = inputs.normal_bf16((16, 256), 1.0, 43)
    c1, s1 = orc.quant_mxfp8(bf16_bits(t))
    c2, s2 = orc.quant_mxfp8(bf16_bits(t * 2))
    assert np.array_equal(c1, c2) and np.array_equal(s2.astype(int), s1.astype(int) + 1)
    z = np.zeros((4, 64), np.uint16)
    cz, sz = orc.quant_mxfp8(z)
    assert not cz.any() and not sz.any()


# ------------------------------------------------------------------ NVFP4
def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """Two 4-bit codes per byte, the lower K index in the low nibble."""
    out = np.empty((packed.shape[0], packed.shape[1] * 2), np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out


def test_nvfp4_two_level_scales(orc):
    x = bf16_bits(inputs.outlier_channel_bf16(64, 256, 51))
    xv = vals(x)
    packed, sc, g = orc.quant_nvfp4(x)
    A = np.abs(xv).max()
    assert abs(float(g) * 2688 - A) <= A * 2.0 ** -22
    dsb = dec_vec(orc.dec_e4m3, sc)
    bmax = np.abs(xv).reshape(64, 16, 16).max(-1)
    assert_nearest(dsb, bmax / 6 / float(g), e4m3_grid(orc), slack=1e-4)
    codes = unpack_e2m1(packed)
    d = np.array([orc.dec_e2m1(c) for c in range(16)])[codes]
    denom = np.repeat(dsb, 16, 1) * float(g)
    ok = denom > 0
    assert_nearest(d[ok], xv[ok] / denom[ok], E2M1_POS, slack=1e-4)
    assert np.all(codes[~ok] & 0x7 == 0)
    # the tensor-amax element: block scale 448, code +-6
    i, k = np.unravel_index(np.argmax(np.abs(xv)), xv.shape)
    assert sc[i, k // 16] == 0x7E and abs(d[i, k]) == 6


def test_nvfp4_packing_nibble_order(orc):
    x = np.zeros((1, 16), np.uint16)
    x[0, 0] = bf16_bits(torch.tensor([[6.0]], dtype=torch.bfloat16))[0, 0]
    x[0, 3] = bf16_bits(torch.tensor([[-3.0]], dtype=torch.bfloat16))[0, 0]
    packed, sc, g = orc.quant_nvfp4(x)
    assert packed[0, 0] == 0x07            # k=0 -> low nibble (+6), k=1 -> high nibble (0)
    assert packed[0, 1] == 0xD0            # k=2 low (0), k=3 high (-3 = 0b1101)
    assert not packed[0, 2:].any()


def test_nvfp4_dequant_close(orc):
    x = bf16_bits(inputs.normal_bf16((32, 128), 1.0, 53))
    xv = vals(x)
    packed, sc, g = orc.quant_nvfp4(x)
    xh = orc.dequant_nvfp4(packed, sc, g)
    unit = np.repeat(dec_vec(orc.dec_e4m3, sc), 16, 1) * float(g)
    bound = half_step(E2M1_POS, xv / unit) * unit * (1 + 1e-4)
    assert np.all(np.abs(xh - xv) <= bound)


def test_nvfp4_exact_bruteforce_small(orc):
    """Every block scale and code against an exact-rational search over all
    UE4M3 and E2M1 codes, on the fp32 values the NVFP4 rule defines:
    q = 448/A and rg = 2688/A, block scale nearest to b*q, element value
    x * (rg / dec(scale)) (0 when the scale decodes to 0), each product or
    quotient one fp32 operation."""
    from test_oracle_codecs import brute_nearest
    e4m3 = [(c, orc.dec_e4m3(c)) for c in range(256) if not math.isnan(orc.dec_e4m3(c))]
    e2m1 = [(c, orc.dec_e2m1(c)) for c in range(16)]
    R, K = 6, 128
    x = bf16_bits(inputs.outlier_channel_bf16(R, K, 57))
    x[5] = bf16_bits(torch.from_numpy(vals(x[5:6]) * 1e-3).to(torch.bfloat16))[0]   # small blocks too
    packed, sc, g = orc.quant_nvfp4(x)
    xv = vals(x).astype(np.float32)                     # bf16 values are exact in fp32
    A = np.float32(np.abs(xv).max())
    q, rg = np.float32(448) / A, np.float32(2688) / A
    assert float(g) == float(A / np.float32(2688))
    codes = unpack_e2m1(packed)
    for i in range(R):
        for blk in range(K // 16):
            seg = xv[i, 16 * blk:16 * blk + 16]
            sb = brute_nearest(float(np.float32(np.abs(seg).max()) * q), e4m3, 448.0, 3)
            assert sc[i, blk] == sb, (i, blk)
            dsb = np.float32(orc.dec_e4m3(sb))
            rb = np.float32(0) if dsb == 0 else rg / dsb
            for k in range(16):
                assert codes[i, 16 * blk + k] == brute_nearest(float(seg[k] * rb), e2m1, 6.0, 1), (i, blk, k)


def _straddle(lo, hi, mids):
    """True where some midpoint m satisfies lo <= m <= hi (the codes may differ)."""
    return np.searchsorted(mids, lo, "left") != np.searchsorted(mids, hi, "right")


def _fragile(v, mids):
    """True where v lies within two fp32 ulps of a code midpoint: there any
    one-ulp change in the steps before the conversion can change the code."""
    lo = np.nextafter(np.nextafter(v, np.float32(0)), np.float32(0))
    hi = np.nextafter(np.nextafter(v, np.float32(np.inf)), np.float32(np.inf))
    return _straddle(lo, hi, mids)


def test_nvfp4_steps_on_fragile_values(orc):
    """Reading R3's fp32 steps, on sweeps of bf16 blocks under fixed tensor
    amaxes: wherever the block value b * fl(448/A) or the element value
    x * fl(fl(2688/A) / dec(sb)) lies within two ulps of a code midpoint, the
    oracle's code is the one an exact-rational search over all codes gives
    for R3's value.  The sweeps include values where the variants b / fl(6 g)
    and x / fl(dec(sb) g) round to another code, so either variant fails."""
    from hard_cases import NVFP4_AMAXES, nvfp4_block_sweep
    from test_oracle_codecs import brute_nearest
    e4m3 = [(c, orc.dec_e4m3(c)) for c in range(256) if not math.isnan(orc.dec_e4m3(c))]
    e2m1 = [(c, orc.dec_e2m1(c)) for c in range(16)]
    pos4 = np.array(sorted({abs(v) for _, v in e4m3}))
    mids4, mids2 = (pos4[1:] + pos4[:-1]) / 2, (E2M1_POS[1:] + E2M1_POS[:-1]) / 2
    dec4 = np.array([orc.dec_e4m3(c) for c in range(256)], np.float32)
    f32 = np.float32
    n_sb = n_el = sep_sb = sep_el = 0
    for A in NVFP4_AMAXES:
        rows = nvfp4_block_sweep(A)
        packed, sc, g = orc.quant_nvfp4(rows)
        x = np.abs(vals(rows).astype(np.float32).reshape(-1, 16))
        b = x.max(1)
        q, rg, gg = f32(448) / f32(A), f32(2688) / f32(A), f32(A) / f32(2688)
        assert f32(g) == gg
        sc = sc.reshape(-1)
        v1, v2 = b * q, b / (f32(6) * gg)
        for i in np.nonzero(_fragile(v1, mids4) | ((v1 != v2) & _straddle(np.minimum(v1, v2),
                                                                        np.maximum(v1, v2), mids4)))[0]:
            c1 = brute_nearest(float(v1[i]), e4m3, 448.0, 3)
            assert sc[i] == c1, (A, i, b[i])
            n_sb += 1
            sep_sb += c1 != brute_nearest(float(v2[i]), e4m3, 448.0, 3)
        dsb = dec4[sc]
        ok = dsb > 0
        rb = np.where(ok, rg / np.where(ok, dsb, f32(1)), f32(0)).astype(np.float32)
        e1 = x * rb[:, None]
        e2 = x / np.where(ok, dsb * gg, f32(1))[:, None]
        codes = unpack_e2m1(packed).reshape(-1, 16)
        cand = ok[:, None] & (_fragile(e1, mids2) | ((e1 != e2) & _straddle(np.minimum(e1, e2),
                                                                           np.maximum(e1, e2), mids2)))
        for i, k in zip(*np.nonzero(cand)):
            c1 = brute_nearest(float(e1[i, k]), e2m1, 6.0, 1)
            assert codes[i, k] == c1, (A, i, k, x[i, k])
            n_el += 1
            sep_el += c1 != brute_nearest(float(e2[i, k]), e2m1, 6.0, 1)
    assert sep_sb > 0 and sep_el > 0, (n_sb, n_el, sep_sb, sep_el)     # the sweeps separate R3 from both variants


def test_nvfp4_worked_blocks(orc):
    """Four blocks worked by hand.  The tensor amax is 448, so 448/A = 1 and
    2688/A = 6 exactly, and g = fl(448/2688).
    Block 0 holds the amax: scale E4M3(448) = 0x7E, multiplier fl(6/448); its
    values sit far from E2M1 ties.  Block 1 (amax 12): scale E4M3(12) = 0x54,
    multiplier 6/12 = 0.5 exactly, so every tie is a true tie and goes to the
    even code; -0.5 -> -0.25 -> -0 keeps its sign.  Block 2 (amax 2^-20): the
    scale rounds to 0 (below half the smallest UE4M3 subnormal), the
    multiplier is 0 and the codes are signed zeros.  Block 3 (amax 2^-8): a
    subnormal scale, code 0x02, multiplier 6/2^-8 = 1536."""
    b0 = [448, 224, 112, -28, 0] + [0] * 11
    b1 = [12, 5, -7, 1.5, 0.5, 10, -3, 2.5, -0.5] + [0] * 7
    b2 = [2.0 ** -20, -2.0 ** -20] + [0] * 14
    b3 = [2.0 ** -8, 2.0 ** -9, -2.0 ** -8] + [0] * 13
    x = bf16_bits(torch.tensor([b0 + b1 + b2 + b3], dtype=torch.bfloat16))
    packed, sc, g = orc.quant_nvfp4(x)
    assert float(g) == float(np.float32(448) / np.float32(2688))
    assert list(sc[0]) == [0x7E, 0x54, 0x00, 0x02]
    codes = list(unpack_e2m1(packed)[0])
    # block 0: 448 -> 6, 224 -> 3, 112 -> 1.5, -28 -> -0.375 -> nearest -0.5
    assert codes[0:16] == [0x7, 0x5, 0x3, 0x9] + [0] * 12
    # block 1 (x 0.5): 6; 2.5 tie 2|3 -> 2; -3.5 tie 3|4 -> 4; 0.75 tie 0.5|1 -> 1;
    # 0.25 tie 0|0.5 -> 0; 5 tie 4|6 -> 4; -1.5; 1.25 tie 1|1.5 -> 1; -0.25 -> -0
    assert codes[16:32] == [0x7, 0x4, 0xE, 0x2, 0x0, 0x6, 0xB, 0x2, 0x8] + [0] * 7
    assert codes[32:48] == [0x0, 0x8] + [0] * 14
    # block 3 (x 1536): 6, 3, -6
    assert codes[48:64] == [0x7, 0x5, 0xF] + [0] * 13
    assert packed[0, 8] == 0x4 << 4 | 0x7       # k = 16 low nibble, k = 17 high nibble


# ------------------------------------------------------------------ MXFP4
def test_mxfp4_shared_exponent_rule(orc):
    # OCP MX rule with the E2M1 element: scale = largest power of two <= amax,
    # divided by 4 (2^2, the exponent of 6, the largest E2M1 binade)
    x = bf16_bits(inputs.outlier_channel_bf16(64, 512, 31))
    xv = vals(x)
    packed, sc = orc.quant_mxfp4(x)
    scale = np.vectorize(orc.dec_e8m0)(sc)
    amax = np.abs(xv).reshape(64, 16, 32).max(-1)
    p2 = np.array([[2.0 ** (math.frexp(a)[1] - 1) for a in row] for row in amax])
    assert np.array_equal(scale, p2 / 4)
    d = dec_vec(orc.dec_e2m1, unpack_e2m1(packed))
    target = xv / np.repeat(scale, 32, 1)                               # exact: power-of-two scaling
    assert_nearest(d, target, E2M1_POS)
    # the amax element lands in [4, 6] (saturating from [6, 8))
    at = np.abs(xv).reshape(64, 16, 32) == amax[..., None]
    dm = np.abs(d).reshape(64, 16, 32)[at]
    assert np.all((dm >= 4) & (dm <= 6))


def test_mxfp4_exact_bruteforce_small(orc):
    from test_oracle_codecs import brute_nearest
    table = [(c, orc.dec_e2m1(c)) for c in range(16)]
    x = bf16_bits(inputs.normal_bf16((2, 64), 3.0, 45))
    packed, sc = orc.quant_mxfp4(x)
    codes = unpack_e2m1(packed)
    xv = vals(x)
    for i in range(2):
        for k in range(64):
            v = xv[i, k] / orc.dec_e8m0(int(sc[i, k // 32]))
            assert codes[i, k] == brute_nearest(v, table, 6.0, 1)


def test_mxfp4_worked_block(orc):
    # a block of exactly representable values at scale 2^3: amax 48 -> floor(log2) 5 -> e = 3;
    # codes are the E2M1 table itself, ties round to the even code, 7 saturates to 6
    vals_ = [48, 32, 24, 16, 12, 8, 4, 0, -48, -4, 20, 40, 2, 6, 56, 1] + [0] * 16
    x = bf16_bits(torch.tensor([vals_], dtype=torch.bfloat16))
    packed, sc = orc.quant_mxfp4(x)
    assert sc[0, 0] == 127 + 3
    codes = unpack_e2m1(packed)[0]
    # 20/8 = 2.5 -> tie between 2 (code 4) and 3 (code 5) -> 4; 40/8 = 5 -> tie 4|6 -> 4 (code 6)
    # 2/8 = 0.25 -> tie 0|0.5 -> 0; 6/8 = 0.75 -> tie 0.5|1 -> 1 (code 2); 56/8 = 7 -> saturates to 6
    # 1/8 = 0.125 -> 0
    want = [0x7, 0x6, 0x5, 0x4, 0x3, 0x2, 0x1, 0x0, 0xF, 0x9, 0x4, 0x6, 0x0, 0x2, 0x7, 0x0] + [0] * 16
    assert list(codes) == want
    assert packed[0, 0] == 0x67            # k=0 -> low nibble (6 -> 0x7), k=1 -> high nibble (4 -> 0x6)
    dq = orc.dequant_mxfp4(packed, sc)[0]
    assert list(dq[:8]) == [48, 32, 24, 16, 12, 8, 4, 0]


def test_mxfp4_scale_offset_from_mxfp8(orc):
    # same MX rule, element exponents 2 (E2M1) and 8 (E4M3): the scale codes differ by 6
    x = bf16_bits(inputs.normal_bf16((8, 256), 1.0, 47))
    _, s4 = orc.quant_mxfp4(x)
    _, s8 = orc.quant_mxfp8(x)
    assert np.array_equal(s4.astype(int), s8.astype(int) + 6)


def test_mxfp4_scale_by_two_and_zero(orc):
    t = inputs.normal_bf16((16, 256), 1.0, 49)
    p1, s1 = orc.quant_mxfp4(bf16_bits(t))
    p2, s2 = orc.quant_mxfp4(bf16_bits(t * 2))
    assert np.array_equal(p1, p2) and np.array_equal(s2.astype(int), s1.astype(int) + 1)
    z = np.zeros((4, 64), np.uint16)
    pz, sz = orc.quant_mxfp4(z)
    assert not pz.any() and not sz.any()


def test_mxfp4_dequant_close(orc):
    x = bf16_bits(inputs.normal_bf16((32, 128), 1.0, 51))
    xv = vals(x)
    packed, sc = orc.quant_mxfp4(x)
    xh = orc.dequant_mxfp4(packed, sc)
    unit = np.repeat(np.vectorize(orc.dec_e8m0)(sc), 32, 1)
    bound = half_step(E2M1_POS, xv / unit) * unit * (1 + 1e-9)
    sat = np.abs(xv / unit) > 6                                        # saturated: off by up to 2 units
    assert np.all(np.abs(xh - xv)[~sat] <= bound[~sat])
    assert np.all(np.abs(xh - xv)[sat] <= 2 * unit[sat])


# ------------------------------------------------------------------ MXFP4 dual-scale (R16)
def _f32_floor_log2(v: float) -> int:
    m, e = math.frexp(v)           # v = m 2^e, 0.5 <= m < 1
    return e - 1


def test_mxfp4_dual_coarse_and_fine_levels(orc):
    """Reading R16: per 512 K the coarse scale is the binary32 nearest to A / 6
    (A the block's amax; 1 for a zero block), and after normalizing by
    fl(6 / A) every 32-element block's largest magnitude lands in [4, 8) times
    its fine power of two (the MX floor rule with the E2M1 exponent 2); the
    element at the block amax encodes to +-6 with fine exponent 0."""
    R, K = 48, 1536
    x = bf16_bits(inputs.outlier_channel_bf16(R, K, 97))
    x[3, 512:1024] = 0                                            # a zero coarse block
    packed, sc, coarse = orc.quant_mxfp4_dual(x)
    assert packed.shape == (R, K // 2) and sc.shape == (R, K // 32) and coarse.shape == (R, K // 512)
    xv = vals(x)
    codes = unpack_e2m1(packed)
    for i in range(R):
        for cb in range(K // 512):
            blk = xv[i, 512 * cb:512 * cb + 512]
            A = np.abs(blk).max()
            c = coarse[i, cb]
            if A == 0:
                assert c == 1.0 and not sc[i, 16 * cb:16 * cb + 16].any()
                assert not (codes[i, 512 * cb:512 * cb + 512] & 7).any()
                continue
            assert Fraction(float(c)) == Fraction(float(np.float32(Fraction(float(A)) / 6)))   # nearest binary32
            r = np.float32(6) / np.float32(A)
            for f in range(16):
                v = (blk[32 * f:32 * f + 32].astype(np.float32) * r).astype(np.float32)
                a = float(np.abs(v).max())
                e = int(sc[i, 16 * cb + f]) - 127
                if a == 0:
                    assert e == -127
                    continue
                assert 4.0 <= a * 2.0 ** -e < 8.0 or e == -127
            k_at = int(np.argmax(np.abs(blk)))
            assert int(sc[i, 16 * cb + k_at // 32]) == 127                  # fine exponent 0
            assert codes[i, 512 * cb + k_at] & 7 == 7                       # |code| = 6


def test_mxfp4_dual_codes_are_nearest_of_the_normalized_values(orc):
    """Codes: the E2M1 value nearest (ties to even) to the exact rational
    fl(x * fl(6 / A)) * 2^-e, saturating at 6, found by a scan of all codes."""
    R, K = 6, 512
    x = rand_bits((R, K), 99)
    packed, sc, coarse = orc.quant_mxfp4_dual(x)
    codes = unpack_e2m1(packed)
    table = [(c, Fraction(orc.dec_e2m1(c))) for c in range(16)]
    xv = vals(x).astype(np.float32)
    for i in range(R):
        r = np.float32(6) / np.float32(np.abs(xv[i]).max())
        for k in range(0, K, 3):
            e = int(sc[i, k // 32]) - 127
            t = Fraction(float(np.float32(xv[i, k] * r))) * Fraction(2) ** -e
            t = max(min(t, Fraction(6)), Fraction(-6))
            best = min(abs(v - t) for _, v in table)
            cands = [c for c, v in table if abs(v - t) == best]
            if len(cands) > 1:
                cands = [c for c in cands if (c & 1) == 0] or cands          # ties to the even mantissa
                if t == 0:
                    cands = [codes[i, k]] if codes[i, k] in (0, 8) else cands
            assert codes[i, k] in cands, (i, k, codes[i, k], cands)


def test_mxfp4_dual_reduces_to_mxfp4_when_the_coarse_scale_is_a_power_of_two(orc):
    """With every 512-block's amax equal to 6 * 2^j the coarse multiplier
    6 / A = 2^-j is exact, so the dual-scale codes are the single-level MXFP4
    codes (reading R11) and every fine exponent is the MXFP4 one minus j."""
    R, K = 16, 1024
    x = rand_bits((R, K), 101)
    xv = vals(x)
    j = np.array([[(i + cb) % 5 - 2 for cb in range(K // 512)] for i in range(R)])
    for i in range(R):
        for cb in range(K // 512):
            blk = xv[i, 512 * cb:512 * cb + 512]
            blk = np.clip(blk, -5.9 * 2.0 ** j[i, cb], 5.9 * 2.0 ** j[i, cb])
            blk[7] = 6.0 * 2.0 ** j[i, cb]
            xv[i, 512 * cb:512 * cb + 512] = blk
    x = bf16_bits(torch.from_numpy(xv).to(torch.bfloat16))
    assert np.array_equal(np.abs(vals(x)).reshape(R, -1, 512).max(-1), 6.0 * 2.0 ** j)
    packed, sc, coarse = orc.quant_mxfp4_dual(x)
    p1, s1 = orc.quant_mxfp4(x)
    assert np.array_equal(packed, p1)
    assert np.array_equal(coarse, (2.0 ** j).astype(np.float32))
    jj = np.repeat(j, 16, axis=1)
    live = s1 > 0
    assert np.array_equal(sc[live].astype(int), s1[live].astype(int) - jj[live])


def test_mxfp4_dual_blocks_are_independent_and_dequant_close(orc):
    R, K = 8, 1536
    x = rand_bits((R, K), 103)
    p1, s1, c1 = orc.quant_mxfp4_dual(x)
    x2 = x.copy()
    x2[5, 512:1024] = bf16_bits(inputs.normal_bf16((1, 512), 300.0, 104))[0]
    p2, s2, c2 = orc.quant_mxfp4_dual(x2)
    changed = np.zeros((R, K // 512), bool)
    changed[5, 1] = True
    assert np.array_equal(c1[~changed], c2[~changed]) and c1[5, 1] != c2[5, 1]
    keep = np.ones((R, K), bool)
    keep[5, 512:1024] = False
    assert np.array_equal(unpack_e2m1(p1)[keep], unpack_e2m1(p2)[keep])
    xh = orc.dequant_mxfp4_dual(p2, s2, c2)
    xv = vals(x2)
    unit = np.repeat(np.vectorize(orc.dec_e8m0)(s2), 32, 1) * np.repeat(c2.astype(np.float64), 512, 1)
    bound = half_step(E2M1_POS, xv / unit) * unit * (1 + 1e-6)
    sat = np.abs(xv / unit) > 6
    assert np.all(np.abs(xh - xv)[~sat] <= bound[~sat])
    assert np.all(np.abs(xh - xv)[sat] <= 2 * unit[sat])


# ------------------------------------------------------------------ int4
def unpack_int4(qweight, qzeros, N, K):
    """GPTQ-style layout: k = 8i + j in bits [4j, 4j+4) of qweight[i, n];
    n = 8i + j in bits [4j, 4j+4) of qzeros[g, i]."""
    qw = qweight.view(np.uint32)
    q = np.empty((K, N), np.int64)
    for j in range(8):
        q[j::8, :] = (qw >> (4 * j)) & 0xF
    qz = qzeros.view(np.uint32)
    z = np.empty((K // 128, N), np.int64)
    for j in range(8):
        z[:, j::8] = (qz >> (4 * j)) & 0xF
    return q, z


def test_int4_rtn_invariants(orc):
    N, K = 64, 384
    w = bf16_bits(inputs.normal_bf16((N, K), 0.02, 61))
    w[5, :128] = bf16_bits(torch.from_numpy(np.abs(vals(w[5:6, :128]))).to(torch.bfloat16))[0]  # all >= 0
    w[6, 128:256] = 0                                                                        # all zero
    wv = vals(w)
    qw, sc, qz = orc.quant_int4_g128(w)
    q, z = unpack_int4(qw, qz, N, K)
    s = vals(sc)                                 # [K/128, N]
    for n in range(N):
        for g in range(K // 128):
            grp = wv[n, g * 128:(g + 1) * 128]
            qq = q[g * 128:(g + 1) * 128, n]
            mn, mx = min(0.0, grp.min()), max(0.0, grp.max())
            sg, zg = s[g, n], z[g, n]
            if mx == mn:
                assert sg == 1.0 and zg == 0 and not qq.any()
                continue
            assert abs(sg - (mx - mn) / 15) <= (mx - mn) / 15 * 2.0 ** -8
            assert 0 <= zg <= 15 and np.all((qq >= 0) & (qq <= 15))
            if mn < 0:
                assert qq[np.argmin(grp)] == 0
            if mn == 0:
                assert zg == 0
            # zero maps exactly: q == z wherever w == 0
            assert np.all(qq[grp == 0] == zg)
            deq = (qq - zg) * sg
            inside = (grp / sg + zg >= -0.5) & (grp / sg + zg <= 15.5)
            assert np.all(np.abs(deq - grp)[inside] <= sg / 2 * (1 + 1e-3))


def test_int4_dequant_and_layout(orc):
    N, K = 16, 256
    w = bf16_bits(inputs.normal_bf16((N, K), 0.02, 63))
    wv = vals(w)
    wv_scaled = wv * np.array([1.0, 100.0])[np.arange(K) // 128][None, :] * (1 + np.arange(N))[:, None]
    wb = bf16_bits(torch.from_numpy(wv_scaled).to(torch.bfloat16))
    wv = vals(wb)
    qw, sc, qz = orc.quant_int4_g128(wb)
    assert qw.shape == (K // 8, N) and sc.shape == (K // 128, N) and qz.shape == (K // 128, N // 8)
    wh = orc.dequant_int4_g128(qw, sc, qz)
    s = vals(sc)
    assert np.all(np.abs(wh - wv) <= np.repeat(s.T, 128, 1) * 0.5 * (1 + 1e-3) + 1e-30)
    q, z = unpack_int4(qw, qz, N, K)
    assert np.array_equal(wh, ((q - np.repeat(z, 128, 0)) * np.repeat(s, 128, 0)).T)


def test_int4_exhaustive_code_roundtrip(orc):
    """Every (q, z) pair survives pack -> unpack: build a weight whose RTN codes
    are known (values already on the grid of a fixed scale) and read them back."""
    N, K = 16, 128
    sgrid = 2.0 ** -6
    rng = np.random.default_rng(0)
    # per column n choose z in 0..15, per k a code q; values (q - z) * s are exact
    z = np.arange(N) % 16
    q = np.array([[(k + 3 * n) % 16 for n in range(N)] for k in range(K)])
    q[0, :] = 0
    q[1, :] = 15                            # force range [(0-z)s, (15-z)s] so s = sgrid
    w = ((q - z[None, :]) * sgrid).T         # [N, K]
    zero_col = z == 0
    wb = bf16_bits(torch.from_numpy(w).to(torch.bfloat16))
    qw, sc, qz = orc.quant_int4_g128(wb)
    qq, zz = unpack_int4(qw, qz, N, K)
    assert np.all(vals(sc) == sgrid)
    assert np.array_equal(zz[0], z)
    assert np.array_equal(qq, q)
    del rng, zero_col


def test_int4_zero_point_and_codes_bruteforce(orc):
    """Given the stored scale s (its value is pinned above), scan all 16
    candidates for z and for every q: z is the candidate nearest to -min/s and
    q - z the offset nearest to x/s, both with 1/s taken once in fp32, exact
    rational distances, and ties to the even integer (-min/s and x/s)."""
    N, K = 8, 256
    w = bf16_bits(inputs.normal_bf16((N, K), 0.02, 65))
    w[1, :128] = bf16_bits(torch.from_numpy(np.abs(vals(w[1:2, :128])) + 0.01).to(torch.bfloat16))[0]
    w[2, 128:] = bf16_bits(torch.from_numpy(-np.abs(vals(w[2:3, 128:]))).to(torch.bfloat16))[0]
    wv = vals(w)
    qw, sc, qz = orc.quant_int4_g128(w)
    q, z = unpack_int4(qw, qz, N, K)
    s = vals(sc)

    def nearest(t: Fraction, cands):
        best = min(abs(c - t) for c in cands)
        tied = [c for c in cands if abs(c - t) == best]
        return tied[0] if len(tied) == 1 else [c for c in tied if c % 2 == 0][0]

    for n in range(N):
        for g in range(K // 128):
            grp = wv[n, g * 128:(g + 1) * 128]
            r = np.float32(1) / np.float32(s[g, n])
            mn = min(0.0, grp.min())
            zt = Fraction(float(np.float32(-mn) * r))
            zb = nearest(zt, range(16))
            assert z[g, n] == zb, (n, g)
            for k in range(0, 128, 3):
                # the offsets q - z that a code can take; outside them the nearest is the end (saturation)
                t = Fraction(float(np.float32(grp[k]) * r))
                assert q[g * 128 + k, n] == nearest(t, range(-zb, 16 - zb)) + zb, (n, g, k)


def test_int4_codes_at_half_steps(orc):
    """Reading R4: q = clamp(rint(x * fl(1/s)) + z) and z = clamp(rint(-min * fl(1/s))),
    1/s taken once in fp32.  On groups of exact half steps (s = 7 * 2^-9, so
    1/s is inexact) x * fl(1/s) lies within an ulp of k + 1/2, where the
    division form x / s would tie to the even integer instead.  The oracle
    follows R4, checked by exact rational distance (round half to even)."""
    from hard_cases import int4_half_step_weight
    w = int4_half_step_weight()
    N, K = w.shape
    qw, sc, qz = orc.quant_int4_g128(w)
    q, z = unpack_int4(qw, qz, N, K)
    f32 = np.float32
    wv = vals(w).astype(np.float32)
    s = vals(sc).astype(np.float32)
    differ = z_differ = 0
    for n in range(N):
        for g in range(K // 128):
            grp = wv[n, 128 * g:128 * g + 128]
            sg = s[g, n]
            assert sg == f32(7.0 / 512)
            r = f32(1) / sg
            mn = f32(-min(0.0, grp.min()))
            zg = min(15, max(0, round(Fraction(float(mn * r)))))
            assert z[g, n] == zg
            z_differ += zg != min(15, max(0, round(Fraction(float(mn)) / Fraction(float(sg)))))
            for k in range(128):
                want = min(15, max(0, round(Fraction(float(grp[k] * r))) + zg))
                assert q[128 * g + k, n] == want, (n, g, k)
                alt = min(15, max(0, round(Fraction(float(grp[k])) / Fraction(float(sg))) + zg))
                differ += want != alt
    assert differ > 0 and z_differ > 0         # the groups do separate R4 from the division forms


def bf16_rne_exact(v: Fraction) -> Fraction:
    """The bf16 value nearest to the exact rational v > 0, ties to an even
    mantissa (8 significant bits), by integer arithmetic."""
    unit = bf16_ulp(v)
    n, rem = divmod(v, unit)
    n = int(n)
    if rem * 2 > unit or (rem * 2 == unit and n % 2):
        n += 1
    return n * unit


def bf16_ulp(v: Fraction) -> Fraction:
    """Spacing of the bf16 values in the binade of v > 0."""
    e = v.numerator.bit_length() - v.denominator.bit_length()
    if Fraction(2) ** e > v:
        e -= 1
    return Fraction(2) ** (e - 7)


def _bf16_of_f32(a: np.ndarray, mode: str) -> np.ndarray:
    """fp32 -> bf16 value by bits: 'rne', 'trunc' or 'half_away'."""
    b = a.astype(np.float32).view(np.uint32).astype(np.uint64)
    lo, kept = b & 0xFFFF, b >> 16
    if mode == "rne":
        kept += (lo > 0x8000) | ((lo == 0x8000) & (kept & 1 == 1))
    elif mode == "half_away":
        kept += lo >= 0x8000
    return (kept.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_int4_scale_rounds_the_range_to_nearest_even(orc):
    """Reading R4's scale step: s = bf16_RNE(fl((max - min) / 15)).  On groups
    whose D / 15 is a bf16 rounding midpoint, or a few fp32 ulps off one
    (tests/hard_cases.py), the oracle's stored scale is the bf16 value nearest
    to the exact rational D / 15 with ties to even; the sweep separates that
    from truncating to bf16, rounding ties away from zero, and multiplying by
    fl(1/15) instead of dividing (each gives another scale on some group)."""
    from hard_cases import int4_scale_tie_weight
    w = int4_scale_tie_weight()
    N, K = w.shape
    qw, sc, qz = orc.quant_int4_g128(w)
    s = vals(sc)[0]
    wv = vals(w)
    mx, mn = np.maximum(wv.max(1), 0.0), np.minimum(wv.min(1), 0.0)
    live = mx > mn
    assert live.sum() >= 3000
    ties = 0
    for n in np.flatnonzero(live):
        d = Fraction(float(mx[n])) - Fraction(float(mn[n]))
        want = bf16_rne_exact(d / 15)
        assert Fraction(float(s[n])) == want, (n, float(mx[n]), float(mn[n]))
        ties += abs(d / 15 - want) == bf16_ulp(d / 15) / 2
    assert ties > 100                          # exact midpoints: the tie rule decides them
    d32 = (mx.astype(np.float32) - mn.astype(np.float32)).astype(np.float32)
    q32 = (d32 / np.float32(15)).astype(np.float32)
    rcp = (d32 * (np.float32(1) / np.float32(15))).astype(np.float32)
    for name, alt in [("trunc", _bf16_of_f32(q32, "trunc")), ("half_away", _bf16_of_f32(q32, "half_away")),
                      ("reciprocal", _bf16_of_f32(rcp, "rne"))]:
        assert (alt[live] != s[live]).any(), name


def test_int4_scale_double_rounding_equals_single(orc):
    """Why R4's scale step has no separate double-rounding reading:
    bf16(fl32(D / 15)) equals bf16(D / 15) rounded once from the exact
    quotient.  D = fl(max - min) and 15 m (m a bf16 midpoint) are both
    multiples of the fp32 ulp of D, so a nonzero D - 15 m is at least that
    ulp, and |D / 15 - m| >= ulp(D) / 15 > ulp(m) / 2: fl32(D / 15) never
    lands on a midpoint that D / 15 itself is not on.  Checked exhaustively
    on every pair of bf16 values max in [1, 4) and min in (-8, 0]."""
    grid = np.concatenate([[0.0], np.arange(256, 512) / 256.0, np.arange(256, 512) / 128.0])
    mxs = grid[grid >= 1]
    mns = -np.concatenate([[0.0], grid[1:], np.arange(256, 512) / 64.0])
    mx, mn = np.meshgrid(mxs, mns, indexing="ij")
    d32 = (mx.astype(np.float32) - mn.astype(np.float32)).astype(np.float32)
    assert np.array_equal(d32.astype(np.float64), mx - mn)          # the range itself is exact here
    twice = _bf16_of_f32((d32 / np.float32(15)).astype(np.float32), "rne")
    for i in range(0, mx.size, 7):
        a, b = mx.flat[i], mn.flat[i]
        assert Fraction(float(twice.flat[i])) == bf16_rne_exact((Fraction(a) - Fraction(b)) / 15), (a, b)
    del orc


# ------------------------------------------------------------------ int4 symmetric (R15)
def test_int4_sym_scale_zero_point_and_range(orc):
    """Reading R15: per group a = max |x|, s = bf16_RNE((a - (-a)) / 15) (the
    bf16 value nearest to the exact 2a / 15, ties to even), zero point 8
    everywhere, a zero group gets s = 1 and codes 8, and zero maps to 8."""
    N, K = 64, 384
    w = rand_bits((N, K), 91, 0.02)
    w[3, 128:256] = 0                                                     # an all-zero group
    w[4, :128] = bf16_bits(torch.from_numpy(np.abs(vals(w[4:5, :128]))).to(torch.bfloat16))[0]   # all >= 0
    w[5, :64] = 0
    qw, sc, qz = orc.quant_int4_g128_sym(w)
    q, z = unpack_int4(qw, qz, N, K)
    assert np.all(z == 8)
    s = vals(sc)
    wv = vals(w)
    for n in range(N):
        for g in range(K // 128):
            grp = wv[n, 128 * g:128 * g + 128]
            a = np.abs(grp).max()
            if a == 0:
                assert s[g, n] == 1.0 and np.all(q[128 * g:128 * g + 128, n] == 8)
                continue
            assert Fraction(float(s[g, n])) == bf16_rne_exact(Fraction(float(a)) * 2 / 15), (n, g)
            qq = q[128 * g:128 * g + 128, n]
            assert np.all(qq[grp == 0] == 8)
            assert np.all((qq >= 0) & (qq <= 15))


def test_int4_sym_codes_bruteforce_and_sign_symmetry(orc):
    """Codes against a scan of the 16 offsets q - 8 in -8 .. 7 with exact
    rational distances to x * fl(1/s) (ties to the even offset, the ends
    saturating), and negating W maps q to 16 - q with the same scales where
    neither side clamps (rint is odd-symmetric; offsets run -8 .. 7)."""
    N, K = 16, 256
    w = bf16_bits(inputs.outlier_channel_bf16(N, K, 93))
    qw, sc, qz = orc.quant_int4_g128_sym(w)
    q, _ = unpack_int4(qw, qz, N, K)
    s = vals(sc).astype(np.float32)
    wv = vals(w).astype(np.float32)

    def nearest(t: Fraction):
        cands = range(-8, 8)
        best = min(abs(c - t) for c in cands)
        tied = [c for c in cands if abs(c - t) == best]
        return tied[0] if len(tied) == 1 else [c for c in tied if c % 2 == 0][0]

    for n in range(N):
        for g in range(K // 128):
            r = np.float32(1) / s[g, n]
            for k in range(0, 128, 5):
                t = Fraction(float(wv[n, 128 * g + k] * r))
                assert q[128 * g + k, n] == nearest(t) + 8, (n, g, k)
    neg = w ^ np.uint16(0x8000)
    qw2, sc2, qz2 = orc.quant_int4_g128_sym(neg)
    q2, _ = unpack_int4(qw2, qz2, N, K)
    assert np.array_equal(sc2, sc)
    mid = (q >= 1) & (q <= 14)                 # rint(x r) in -7 .. 6: neither side clamps
    assert np.array_equal(q2[mid], 16 - q[mid])
    assert np.all(q2[q == 0] == 15)            # -8 turns into +8, which clamps to 7
    assert np.all((q2[q == 15] == 1) | (q2[q == 15] == 0))   # +7, or +8 clamped, turns into -7 or -8


def test_int4_sym_codes_at_half_steps(orc):
    """Reading R15's fp32 steps: q = clamp(rint(x * fl(1/s)) + 8).  On groups
    of exact half steps of s = 7 * 2^-9 (tests/hard_cases.py) x * fl(1/s)
    lies next to k + 1/2; the oracle's codes are the exact nearest integers of
    that product (ties to even) plus 8, and dividing, x / s, would give other
    codes on some of them."""
    from hard_cases import int4_sym_half_step_weight
    w = int4_sym_half_step_weight()
    N, K = w.shape
    qw, sc, qz = orc.quant_int4_g128_sym(w)
    q, z = unpack_int4(qw, qz, N, K)
    assert np.all(z == 8)
    s = vals(sc).astype(np.float32)
    wv = vals(w).astype(np.float32)
    differ = 0
    for n in range(N):
        for g in range(K // 128):
            assert s[g, n] == np.float32(7.0 / 512)
            r = np.float32(1) / s[g, n]
            for k in range(128):
                x = wv[n, 128 * g + k]
                want = min(15, max(0, round(Fraction(float(x * r))) + 8))
                assert q[128 * g + k, n] == want, (n, g, k)
                differ += want != min(15, max(0, round(Fraction(float(x)) / Fraction(float(s[g, n]))) + 8))
    assert differ > 0


def test_int4_sym_dequant_within_half_step(orc):
    """(q - 8) s is within s/2 of x wherever x / s + 8 is inside [-0.5, 15.5];
    only the top end (x near +a, offset 7.5) can saturate, by one step."""
    N, K = 32, 512
    w = bf16_bits(inputs.normal_bf16((N, K), 0.02, 95))
    qw, sc, qz = orc.quant_int4_g128_sym(w)
    wh = orc.dequant_int4_g128(qw, sc, qz)
    wv = vals(w)
    s = np.repeat(vals(sc).T, 128, 1)
    err = np.abs(wh - wv)
    inside = (wv / s + 8 >= -0.5) & (wv / s + 8 <= 15.5)
    assert np.all(err[inside] <= s[inside] / 2 * (1 + 1e-3))
    assert np.all(err[~inside] <= s[~inside] * (1 + 1e-3))


# ------------------------------------------------------------------ INT8 per row
def test_int8_worked_rows_ties_and_saturation(orc):
    """Rows chosen so that 127/amax is a power of two: x * r is exact and the
    expected codes follow from the definition by hand (ties to even)."""
    row1 = [127.0, 0.5, 1.5, 2.5, -0.5, -1.5, 126.5, -127.0]      # amax 127: r = 1
    row2 = [254.0, 3.0, 5.0, -7.0, 1.0, -254.0, 0.0, 253.0]       # amax 254: r = 1/2
    x = bf16_bits(torch.tensor([row1, row2], dtype=torch.bfloat16))
    codes, s = orc.quant_int8_row(x)
    assert codes.dtype == np.int8
    assert codes[0].tolist() == [127, 0, 2, 2, 0, -2, 126, -127]
    assert codes[1].tolist() == [127, 2, 2, -4, 0, -127, 0, 126]
    assert s.tolist() == [1.0, 2.0]


def test_int8_codes_follow_the_reciprocal_form(orc):
    """Reading R13: code = clamp(rint(x * fl(127 / amax))).  On a sweep of rows
    led by their amax (tests/hard_cases.py), wherever x * fl(127/amax) lies
    within two ulps of a half-integer the oracle's code is the nearest integer
    (half to even) by exact rational distance; the sweep includes rows where
    the division form x / fl(amax / 127) rounds to another integer."""
    from hard_cases import row_amax_sweep
    rows = row_amax_sweep()
    codes, scales = orc.quant_int8_row(rows)
    f32 = np.float32
    x = vals(rows).astype(np.float32)
    a = np.abs(x).max(1)
    r = (f32(127) / a).astype(np.float32)
    assert np.array_equal(scales, (a / f32(127)).astype(np.float32))
    v = x * r[:, None]
    lo = np.nextafter(np.nextafter(v, f32(-np.inf)), f32(-np.inf))
    hi = np.nextafter(np.nextafter(v, f32(np.inf)), f32(np.inf))
    fragile = np.floor(lo - f32(0.5)) != np.floor(hi - f32(0.5))        # a half-integer in [lo, hi]
    alt = np.rint(x / (a / f32(127))[:, None])
    checked = separated = 0
    c = codes.view(np.int8).astype(np.int64)
    for i, k in zip(*np.nonzero(fragile)):
        want = min(127, max(-127, round(Fraction(float(v[i, k])))))
        assert c[i, k] == want, (i, k, x[i, k])
        checked += 1
        separated += want != alt[i, k]
    assert checked > 500 and separated > 0


def test_int8_amax_maps_to_127_and_codes_are_nearest(orc):
    R, K = 48, 384
    x = bf16_bits(inputs.outlier_channel_bf16(R, K, 91))
    xv = vals(x)
    codes, s = orc.quant_int8_row(x)
    q = codes.astype(np.float64)
    a = np.abs(xv).max(1)
    assert np.all(np.abs(s.astype(np.float64) * 127 - a) <= a * 2.0 ** -22)   # s = amax/127 to binary32
    for i in range(R):
        assert np.all(np.abs(q[i][np.abs(xv[i]) == a[i]]) == 127)
    target = xv * (127.0 / a)[:, None]
    assert np.all(np.abs(q - target) <= 0.5 + 1e-4) and np.all(np.abs(q) <= 127)


def test_int8_zero_row_scaling_and_sign(orc):
    x = rand_bits((6, 256), 93)
    x[2] = 0
    c1, s1 = orc.quant_int8_row(x)
    assert not c1[2].any() and s1[2] == 1.0
    x2 = bf16_bits(torch.from_numpy(vals(x) * 2.0).to(torch.bfloat16))
    c2, s2 = orc.quant_int8_row(x2)
    keep = np.arange(6) != 2
    assert np.array_equal(c1, c2) and np.array_equal(s2[keep], 2 * s1[keep])
    c3, s3 = orc.quant_int8_row(x ^ np.uint16(0x8000))
    assert np.array_equal(c3, -c1) and np.array_equal(s3, s1)


def test_int8_rows_are_independent_and_dequant_close(orc):
    x = rand_bits((8, 512), 95)
    c1, s1 = orc.quant_int8_row(x)
    x2 = x.copy()
    x2[4] = bf16_bits(inputs.normal_bf16((1, 512), 50.0, 96))[0]
    c2, s2 = orc.quant_int8_row(x2)
    keep = np.arange(8) != 4
    assert np.array_equal(c1[keep], c2[keep]) and np.array_equal(s1[keep], s2[keep]) and s1[4] != s2[4]
    # rows 10^k apart: a scale applied to the wrong row misses by orders of magnitude
    xv = vals(x) * (10.0 ** np.arange(8))[:, None]
    xb = bf16_bits(torch.from_numpy(xv).to(torch.bfloat16))
    c, sc = orc.quant_int8_row(xb)
    xh = orc.dequant_int8_row(c, sc)
    assert np.all(np.abs(xh - vals(xb)) <= sc.astype(np.float64)[:, None] * 0.5 * (1 + 1e-5))


def test_int8_gemm_is_scaled_integer_product(orc):
    """Over INT8 operands the GEMM reference (float64 matmul of dequantized
    values) equals s_x[m] * s_w[n] times the exact int64 dot product of the codes."""
    M, N, K = 24, 40, 256
    cx, sx = orc.quant_int8_row(rand_bits((M, K), 97))
    cw, sw = orc.quant_int8_row(rand_bits((N, K), 98, 0.02))
    y = orc.gemm_ref(orc.dequant_int8_row(cx, sx), orc.dequant_int8_row(cw, sw))
    ss = sx.astype(np.float64)[:, None] * sw.astype(np.float64)[None, :]
    expect = ss * (cx.astype(np.int64) @ cw.astype(np.int64).T)
    # each float64 product of two dequantized values rounds once (62 bits)
    mag = ss * (np.abs(cx.astype(np.int64)) @ np.abs(cw.astype(np.int64)).T)
    assert np.all(np.abs(y - expect) <= mag * K * 2.0 ** -52)


# ------------------------------------------------------------------ every format
MONOTONE_CASES = {
    # name: (quantize, dequantize, length of the sorted runs along K)
    "fp8_tensor": ("quant_fp8_tensor", "dequant_fp8_tensor", 64),
    "fp8_token": ("quant_fp8_token", "dequant_fp8_token", 64),
    "fp8_block128": ("quant_fp8_block128", "dequant_fp8_block128", 128),
    "fp8_group128": ("quant_fp8_group128", "dequant_fp8_group128", 128),
    "mxfp8": ("quant_mxfp8", "dequant_mxfp8", 32),
    "mxfp4": ("quant_mxfp4", "dequant_mxfp4", 32),
    "nvfp4": ("quant_nvfp4", "dequant_nvfp4", 16),
    "int8_row": ("quant_int8_row", "dequant_int8_row", 64),
    "int4_g128": ("quant_int4_g128", "dequant_int4_g128", 128),
    "int4_g128_sym": ("quant_int4_g128_sym", "dequant_int4_g128", 128),
    "mxfp4_dual": ("quant_mxfp4_dual", "dequant_mxfp4_dual", 32),
}


@pytest.mark.parametrize("name", sorted(MONOTONE_CASES))
def test_dequant_of_quant_is_monotone(orc, name):
    """Within one granule the scale is fixed and rounding to a grid is
    monotone, so dequant(quant(x)) never decreases along sorted x.  Each run
    is sorted in place: no granule's amax (nor min, for int4) changes.  A
    wrong sign bit, a swapped nibble pair or a misplaced scale breaks it."""
    qname, dname, run = MONOTONE_CASES[name]
    R, K = 128, 512
    x = bf16_bits(inputs.outlier_channel_bf16(R, K, 67))
    order = np.argsort(vals(x).reshape(R, K // run, run), axis=-1, kind="stable")
    xs = np.take_along_axis(x.reshape(R, K // run, run), order, axis=-1).reshape(R, K)
    deq = getattr(orc, dname)(*getattr(orc, qname)(xs))
    assert deq.shape == (R, K)
    assert np.all(np.diff(deq.reshape(R, K // run, run), axis=-1) >= 0)
    # and the runs hold values of both signs, so the check spans the sign boundary
    assert (vals(xs) < 0).any() and (vals(xs) > 0).any()


# ------------------------------------------------------------------ GEMM reference
def test_gemm_ref_exact_rational_tiny(orc):
    rng = np.random.default_rng(1)
    for (M, N, K) in [(1, 1, 1), (3, 5, 7), (17, 9, 32), (32, 32, 32)]:
        xb = bf16_bits(inputs.normal_bf16((M, K), 1.0, 100 + M))
        wb = bf16_bits(inputs.normal_bf16((N, K), 1.0, 200 + N))
        cx, sx = orc.quant_fp8_token(xb)
        xh = orc.dequant_fp8_token(cx, sx)
        wh = vals(wb)
        alpha = 0.75
        bias = rng.standard_normal(N)
        y = orc.gemm_ref(xh, wh, alpha=alpha, bias=bias)
        for m in range(M):
            for n in range(N):
                exact = Fraction(alpha) * sum(Fraction(float(xh[m, k])) * Fraction(float(wh[n, k]))
                                              for k in range(K)) + Fraction(float(bias[n]))
                assert abs(Fraction(float(y[m, n])) - exact) <= abs(exact) * Fraction(1, 2 ** 40) + Fraction(1, 2 ** 60)


def test_gemm_ref_orientation(orc):
    """Y = X W^T: Y[m, n] pairs row m of X with row n of W (nn.Linear layout)."""
    X = np.zeros((2, 3)); X[1, 2] = 1.0
    W = np.zeros((4, 3)); W[3, 2] = 5.0
    Y = orc.gemm_ref(X, W)
    assert Y.shape == (2, 4) and Y[1, 3] == 5.0 and np.count_nonzero(Y) == 1


def test_gemm_metrics_and_pass_rule(orc):
    rng = np.random.default_rng(2)
    y = rng.standard_normal((64, 64))
    ok, m = orc.gemm_pass(orc.bf16_round(y), y)
    assert ok and m["relative_l2"] == pytest.approx(m["bf16_floor"])
    ok, m = orc.gemm_pass(y * (1 + 5e-3), y)
    assert not ok and m["relative_l2"] == pytest.approx(5e-3)
    assert m["cosine"] == pytest.approx(1.0)
