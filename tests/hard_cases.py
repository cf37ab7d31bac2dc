"""Constructed inputs on which two readings of a rounding rule give different
codes (test inputs only: no expected values are computed here).

NVFP4: `nvfp4_block_sweep` enumerates bf16 blocks under a fixed tensor amax,
so that the block scale b * fl(448 / A) and the element value
x * fl(fl(2688 / A) / dec(scale)) meet, somewhere in the sweep, the rare
values where a variant of those steps (b / (6 g), x / (dec(scale) g)) rounds
to another code.

FP8 granules encode x * r with r = fl(448 / amax), one fp32 reciprocal per
granule.  Dividing instead, x / fl(amax / 448), gives the same code almost
everywhere; the pairs below are where it does not.  With amax = 7 t 2^j
(t odd), amax / 448 = t 2^j / 64 is exact in fp32 while 448 / amax is not,
and x = m amax / 448 for an E4M3 midpoint m is a bf16 value.  So the
division lands exactly on the midpoint (and ties to the even code), while
the rounded reciprocal can move the product off it.
"""
import math

import numpy as np


def _is_bf16(v: float) -> bool:
    return (int(np.array([v], np.float32).view(np.uint32)[0]) & 0xFFFF) == 0


def fp8_reciprocal_candidates(e4m3_values):
    """(amax, x) pairs, amax >= x > 0, both bf16, with x * 448 / amax an E4M3
    midpoint.  `e4m3_values` are the decoded E4M3 codes (NaNs ignored)."""
    pos = sorted({abs(v) for v in e4m3_values if not math.isnan(v)})
    mids = [(lo + hi) / 2 for lo, hi in zip(pos[:-1], pos[1:])]
    out = []
    for t in range(1, 37, 2):
        for j in range(-6, 6):
            a = 7.0 * t * 2.0 ** j
            if not _is_bf16(a):
                continue
            for m in mids:
                x = m * a / 448
                if 0 < x <= a and _is_bf16(x):
                    out.append((a, x))
    return out


def rows_of_pairs(pairs, K: int) -> np.ndarray:
    """bf16 bits of rows [amax, x, 0, ...] (K elements each), one row per pair."""
    rows = np.zeros((len(pairs), K), np.float32)
    for i, (a, x) in enumerate(pairs):
        rows[i, 0], rows[i, 1] = a, x
    return (rows.view(np.uint32) >> 16).astype(np.uint16)


def bf16_grid(lo_exp: int, hi_exp: int) -> np.ndarray:
    """Every positive bf16 value in [2^lo_exp, 2^hi_exp), ascending, as float32."""
    e = np.arange(lo_exp + 127, hi_exp + 127, dtype=np.uint32)
    bits = ((e[:, None] << 7) | np.arange(128, dtype=np.uint32)[None, :]).ravel() << 16
    return bits.view(np.float32)


# tensor amaxes (bf16) under which the NVFP4 steps separate from their variants
NVFP4_AMAXES = (13.0, 2.046875, 4.71875, 0.171875, 5.1875)


def nvfp4_block_sweep(A: float, binades: int = 5, K: int = 256) -> np.ndarray:
    """bf16 bits of one tensor whose amax is A: a block [A, 0, ...], then for
    every bf16 b from 2^(floor(log2 A) - binades) up to A, blocks led by b and
    filled with the bf16 values x <= b of that range in order, so that each
    (b, x) pair appears once.  Rows of K elements (K / 16 blocks), padded with
    zero blocks."""
    lo = int(np.floor(np.log2(A))) - binades
    grid = bf16_grid(lo, lo + binades + 1)
    bs = grid[grid <= A]
    blocks = [np.array([A] + [0.0] * 15, np.float32)]
    for b in bs:
        xs = grid[grid <= b]
        for i in range(0, len(xs), 15):
            chunk = xs[i:i + 15]
            blk = np.zeros(16, np.float32)
            blk[0], blk[1:1 + len(chunk)] = b, chunk
            blocks.append(blk)
    per_row = K // 16
    n = -(-len(blocks) // per_row) * per_row
    out = np.zeros((n, 16), np.float32)
    out[:len(blocks)] = np.stack(blocks)
    return (out.reshape(-1, K).view(np.uint32) >> 16).astype(np.uint16)


def int4_half_step_weight(N: int = 64, s: float = 7.0 / 512) -> np.ndarray:
    """bf16 bits of W [N, 256] (two groups of 128 per channel) in which every
    group spans exactly 15 steps of s: its minimum is -z0 s with z0 in
    {0, 1, 2, 4, 8} (even channels) or -(z0 + 1/2) s with z0 in
    {3, 6, 9, 12, 14} (odd channels), and its maximum 15 steps above, so its
    step is exactly s.  The other values are (k + 1/2) s for
    every half step inside the range.  With s = 7 * 2^-9 all of them are bf16
    values, and 1/s is inexact in fp32, so x * fl(1/s) often rounds to a value
    next to the half-integer k + 1/2 instead of onto it."""
    w = np.zeros((N, 256), np.float32)
    for n in range(N):
        for g in range(2):
            if n % 2:
                # the minimum itself half a step off the grid: -min / s = z0 + 1/2 sits next to a tie too
                z0 = (6, 12, 14, 3, 9)[(n + 3 * g) % 5]
                lo, hi = -(z0 + 0.5) * s, (14.5 - z0) * s
            else:
                z0 = (0, 1, 2, 4, 8)[(n + 3 * g) % 5]
                lo, hi = -z0 * s, (15 - z0) * s
            vals = [lo, hi] + [(k + 0.5) * s for k in range(-z0, 15 - z0) if lo <= (k + 0.5) * s <= hi]
            row = np.resize(np.array(vals, np.float32), 128)
            w[n, 128 * g:128 * g + 128] = row
    bits = w.view(np.uint32)
    assert not (bits & 0xFFFF).any()                    # every value is a bf16 value
    return (bits >> 16).astype(np.uint16)


def row_amax_sweep(lo_exp: int = -4, hi_exp: int = 8, stride: int = 3, K: int = 256) -> np.ndarray:
    """bf16 bits of rows that each start with their amax a and hold bf16 values
    x <= a after it: for every `stride`-th bf16 a in [2^lo_exp, 2^hi_exp),
    every bf16 x <= a of that range appears once (K - 1 per row).  Per-row
    encoders multiply x by one rounded reciprocal of a, so the sweep meets the
    values where that product sits next to a rounding tie."""
    grid = bf16_grid(lo_exp, hi_exp)
    rows = []
    for a in grid[::stride]:
        xs = grid[grid <= a]
        for i in range(0, len(xs), K - 1):
            row = np.zeros(K, np.float32)
            chunk = xs[i:i + K - 1]
            row[0], row[1:1 + len(chunk)] = a, chunk
            rows.append(row)
    return (np.stack(rows).view(np.uint32) >> 16).astype(np.uint16)


def tiles_of_pairs(pairs, n_tiles: int = 64) -> np.ndarray:
    """bf16 bits of W [128, 128 * n] holding one pair per 128 x 128 tile:
    amax at the tile's (0, 0) and x at (0, 1), zeros elsewhere."""
    pairs = list(pairs)[:n_tiles]
    w = np.zeros((128, 128 * len(pairs)), np.float32)
    for t, (a, x) in enumerate(pairs):
        w[0, 128 * t], w[0, 128 * t + 1] = a, x
    return (w.view(np.uint32) >> 16).astype(np.uint16)


def int4_scale_tie_weight(binades=(-20, -7, -3, 0, 4)) -> np.ndarray:
    """bf16 bits of W [N, 128] (one int4 group per channel) whose range
    D = max - min puts D / 15 on a bf16 rounding midpoint or within a few
    fp32 ulps of one.  For a midpoint m = (257 + 2j) 2^(e-8) of binade e,
    T = 15 (257 + 2j) has at most 13 significant bits; it is split into
    hi = T with its low 5 bits cleared (at most 8 bits) and lo = T - hi (at
    most 5 bits), both bf16 values once scaled by 2^(e-8).  Each (e, j) gives
    six groups: max = hi and min = -lo, or max = lo and min = -hi, each with
    lo as is (D / 15 = m exactly) or with lo * 8 -+ 1 in units of 2^(e-11)
    (D / 15 = m -+ 2^(e-11) / 15, just off the midpoint).  The other values
    of a group are zeros and min / 2."""
    groups = []
    for e in binades:
        unit = 2.0 ** (e - 8)
        for j in range(128):
            T = 15 * (257 + 2 * j)
            hi = T & ~0x1F
            lo = T - hi
            for lo_v in (lo * unit, (8 * lo - 1) * unit / 8, (8 * lo + 1) * unit / 8):
                for mx, mn in ((hi * unit, -lo_v), (lo_v, -hi * unit)):
                    g = np.zeros(128, np.float32)
                    g[0], g[1], g[2] = mx, mn, mn / 2
                    groups.append(g)
    w = np.stack(groups)
    w = np.concatenate([w, np.zeros(((-len(w)) % 8, 128), np.float32)])   # N multiple of 8
    bits = w.view(np.uint32)
    assert not (bits & 0xFFFF).any()                    # every value is a bf16 value
    return (bits >> 16).astype(np.uint16)


def int4_sym_half_step_weight(N: int = 64, s: float = 7.0 / 512) -> np.ndarray:
    """bf16 bits of W [N, 256] for the symmetric int4 rule: every group holds
    its amax a = 7.5 s (so 2a / 15 = s exactly, a bf16 value, and 1/s is
    inexact in fp32), with the sign of a alternating over channels, and
    then the half steps (k + 1/2) s for k = -8 .. 7 and the whole steps k s
    for k = -7 .. 7 in a per-group rotation.  x * fl(1/s) then often lands
    next to the half-integer k + 1/2 instead of on it."""
    w = np.zeros((N, 256), np.float32)
    halves = [(k + 0.5) * s for k in range(-8, 8)]
    wholes = [k * s for k in range(-7, 8)]
    for n in range(N):
        for g in range(2):
            vals = halves + wholes
            rot = (3 * n + 5 * g) % len(vals)
            vals = vals[rot:] + vals[:rot]
            row = np.resize(np.array(vals, np.float32), 128)
            row[0] = 7.5 * s if (n + g) % 2 == 0 else -7.5 * s
            w[n, 128 * g:128 * g + 128] = row
    bits = w.view(np.uint32)
    assert not (bits & 0xFFFF).any()                    # every value is a bf16 value
    return (bits >> 16).astype(np.uint16)
