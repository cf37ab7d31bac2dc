"""Constructed inputs on which two readings of a rounding rule give different
codes (test inputs only: no expected values are computed here).

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
