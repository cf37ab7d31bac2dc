"""Host checks of the bit-level arithmetic the kernels rely on, written from
the IEEE formats (numpy emulates the half-precision operations exactly).

- INT8 GEMM: a code q becomes the fp16 value of the same integer as
  bits(0x6400 | (q ^ 0x80)) - 1152.
- W4A16: codes q and zero point z give bf16(0x4300 | q) - bf16(0x4300 | z),
  taken two at a time from bits [4j, 4j + 4) and [4j + 16, 4j + 20).
- The warp-level W4A16 kernel: lane q's A-fragment positions and B-fragment
  positions name the same K index for every logical k of an m16n8k16 step.
"""
import numpy as np


def f16(bits):
    return np.array(bits, dtype=np.uint16).view(np.float16)


def bf16_value(bits):
    return float(np.array([int(bits) << 16], dtype=np.uint32).view(np.float32)[0])


def test_int8_to_fp16_is_exact_for_every_code():
    q = np.arange(-128, 128, dtype=np.int32)
    u = (q & 0xFF) ^ 0x80                       # the byte with its top bit flipped: q + 128
    biased = f16(0x6400 | u)                    # 1024 + u, exact (11-bit significand)
    out = biased - np.float16(1152.0)           # one fp16 subtraction per value
    assert out.dtype == np.float16
    assert np.array_equal(out.astype(np.int32), q)
    assert np.float16(1152.0).view(np.uint16) == 0x6480


def test_int4_pairs_to_bf16_are_exact_for_every_code_and_zero_point():
    for z in range(16):
        for q in range(16):
            a = bf16_value(0x4300 | q)          # 128 + q
            b = bf16_value(0x4300 | z)          # 128 + z
            assert a == 128 + q and b == 128 + z
            assert a - b == q - z               # exact in bf16: |q - z| <= 15
    # the pair extraction: bits [4j, 4j+4) and [4j+16, 4j+20) of one word
    for w in (0x76543210, 0xA5F30C69, 0xFFFFFFFF, 0x00000000):
        codes = [(w >> (4 * i)) & 0xF for i in range(8)]
        for j in range(4):
            v = ((w >> (4 * j)) & 0x000F000F) | 0x43004300
            lo, hi = v & 0xFFFF, v >> 16
            assert (lo, hi) == (0x4300 | codes[j], 0x4300 | codes[j + 4])


def test_warp_mma_k_order_matches_between_operands():
    """m16n8k16: lane q holds A (and B) logical k = 2q, 2q+1 in its first
    register and 2q+8, 2q+9 in its second.  The kernel stages X with each 8-K
    octet in the order 0 4 1 5 2 6 3 7 and reads positions 4q .. 4q+3 of the
    16-K step; it dequantizes W from octet q // 2 as pairs (j, j+4), (j+1, j+5),
    j = 2 (q % 2).  Both must name the same physical k for every logical k."""
    perm = [0, 4, 1, 5, 2, 6, 3, 7]
    staged = [8 * (p // 8) + perm[p % 8] for p in range(16)]   # physical k at staged position p
    for q in range(4):
        a_phys = {2 * q: staged[4 * q], 2 * q + 1: staged[4 * q + 1],
                  2 * q + 8: staged[4 * q + 2], 2 * q + 9: staged[4 * q + 3]}
        o, j = q // 2, 2 * (q % 2)
        b_phys = {2 * q: 8 * o + j, 2 * q + 1: 8 * o + j + 4,
                  2 * q + 8: 8 * o + j + 1, 2 * q + 9: 8 * o + j + 5}
        assert a_phys == b_phys
    # and the 16 logical k of a step cover the 16 physical k once
    covered = sorted(8 * (q // 2) + 2 * (q % 2) + d for q in range(4) for d in (0, 4, 1, 5))
    assert covered == list(range(16))
