"""Host checks of the bit-level arithmetic the kernels rely on, written from
the IEEE formats (numpy emulates the half-precision operations exactly).

- INT8 GEMM: a code q becomes the fp16 value of the same integer as
  bits(0x6400 | (q ^ 0x80)) - 1152.
- W4A16: codes q and zero point z give bf16(0x4300 | q) - bf16(0x4300 | z),
  taken two at a time from bits [4j, 4j + 4) and [4j + 16, 4j + 20).
- The warp-level W4A16 kernel: lane q's A-fragment positions and B-fragment
  positions name the same K index for every logical k of an m16n8k16 step.
- The grids: the GEMM tile raster, the quantizers' task walks and tile grids,
  the tensor-core scale tiling and the W4A16 split-K partitions each cover
  their outputs exactly once.
"""
from collections import Counter

import numpy as np
import pytest


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


# ---------------------------------------------------------------- grid coverage
# The kernels' index math restated on the host (each function names the kernel
# it follows): every output element, tile and K group is visited exactly once,
# for the workloads' shapes and for ragged ones.
SMS = 152


def cdiv(a, b):
    return -(-a // b)


def tile_coords(t, tiles_m, tiles_n, BN, BM=128, GM=16):
    """gemm_tc.cu, tile_coords: bands of 16 row blocks, rows first inside a band."""
    band = t // (GM * tiles_n)
    first_m = band * GM
    gm = min(GM, tiles_m - first_m)
    idx = t - band * GM * tiles_n
    return (first_m + idx % gm) * BM, (idx // gm) * BN


@pytest.mark.parametrize("M,N", [(128, 1024), (4096, 12288), (32768, 3072), (20280, 13824), (20280, 5120),
                                 (333, 1040), (1, 72), (2100, 640)])
def test_gemm_raster_visits_every_output_tile_once(M, N):
    BN = 256
    tm, tn = cdiv(M, 128), cdiv(N, BN)
    got = [tile_coords(t, tm, tn, BN) for t in range(tm * tn)]
    assert sorted(got) == [(i * 128, j * BN) for i in range(tm) for j in range(tn)]
    # the persistent loop (tile = blockIdx.x; tile += gridDim.x) hands each index to one CTA
    grid = min(tm * tn, SMS)
    owners = Counter(t for b in range(grid) for t in range(b, tm * tn, grid))
    assert set(owners.values()) == {1} and len(owners) == tm * tn


def task_pos(t, total, tpr, nvr, lane):
    """quant.cu, task_pos: task t is 32 consecutive 16-byte vectors of one row."""
    if t >= total:
        return None
    row = t // tpr
    c = (t - row * tpr) * 32 + lane
    return (row, c) if c < nvr else None


def task_walk(rows, K, grid, unroll=4):
    """The walk of k_amax_partial and k_fp8_tensor_encode: warp w0 = 8 * block
    + warp takes tasks t + u * warps for u < unroll, then steps by warps *
    unroll."""
    nvr = K // 8
    tpr = cdiv(nvr, 32)
    total = rows * tpr
    warps = grid * 8
    seen = Counter()
    for w0 in range(warps):
        for t in range(w0, total, warps * unroll):
            for u in range(unroll):
                for lane in range(32):
                    p = task_pos(t + u * warps, total, tpr, nvr, lane)
                    if p is not None:
                        seen[p] += 1
    return seen, nvr


def task_grid_once(rows, K, unroll=4):
    return max(1, cdiv(rows * cdiv(K // 8, 32), 8 * unroll))


def task_grid_persistent(rows, K, unroll=4):
    return max(1, min(cdiv(rows * cdiv(K // 8, 32), 8 * unroll), SMS * 8))


def amax_partials(rows, K):
    return max(1, min(cdiv(rows * (K // 8), 1024), 1024))


@pytest.mark.parametrize("rows,K", [(333, 1040), (128, 1024), (3, 8), (200, 512), (1, 20480), (130, 264)])
def test_task_walks_cover_every_vector_once(rows, K):
    for grid in {task_grid_once(rows, K), task_grid_persistent(rows, K), amax_partials(rows, K), 1, 3}:
        seen, nvr = task_walk(rows, K, grid)
        assert len(seen) == rows * nvr and set(seen.values()) == {1}, grid
        assert all(r < rows and c < nvr for r, c in seen)
    # the one-round grid needs no second round
    g = task_grid_once(rows, K)
    assert g * 8 * 4 >= rows * cdiv(K // 8, 32)


CHUNK_U = 4
CHUNK = 32 * CHUNK_U


def chunk_grid(rows, K):
    """quant.cu, chunk_grid: row blocks of 8 along x, 1024-element chunks along y."""
    return cdiv(rows, 8), cdiv(K // 8, CHUNK)


def chunk_vectors(bx, by, warp, lane, rows, K):
    """k_fp8_group128 / k_mx: warp `warp` of CTA (bx, by) owns row 8 bx + warp and
    the vectors by * CHUNK + lane + 32 u, u < CHUNK_U, that lie in the row."""
    row = bx * 8 + warp
    if row >= rows:
        return []
    nvr = K // 8
    return [(row, c) for c in (by * CHUNK + lane + 32 * u for u in range(CHUNK_U)) if c < nvr]


@pytest.mark.parametrize("rows,K", [(333, 1040), (128, 1024), (3, 32), (200, 512), (1, 20480), (130, 5120),
                                    (20352, 128)])
def test_chunk_walks_cover_every_vector_once(rows, K):
    gx, gy = chunk_grid(rows, K)
    seen = Counter(v for bx in range(gx) for by in range(gy) for w in range(8) for ln in range(32)
                   for v in chunk_vectors(bx, by, w, ln, rows, K))
    assert len(seen) == rows * (K // 8) and set(seen.values()) == {1}
    # the persistent NVFP4 encode pass: CTA b takes ids b, b + grid, ...; id -> (id // gy, id % gy)
    for grid in {1, 7, min(gx * gy, SMS * 8)}:
        ids = Counter(i for b in range(grid) for i in range(b, gx * gy, grid))
        assert set(ids.values()) == {1} and len(ids) == gx * gy
        assert sorted(divmod(i, gy) for i in ids) == [(x, y) for x in range(gx) for y in range(gy)]
    # a granule never straddles a chunk: 1024 elements hold whole 16-, 32- and 128-element granules
    assert CHUNK * 8 % 128 == 0


def test_block128_and_int4_grids_cover_their_tiles():
    # k_fp8_block128: CTA b -> tile (b // (K/128), b % (K/128)); thread t -> rows t/16 + 16 i, vector t % 16
    rows, K = 384, 640
    kt = K // 128
    seen = Counter()
    for b in range((rows // 128) * kt):
        bi, bj = b // kt, b - (b // kt) * kt
        for t in range(256):
            for i in range(8):
                seen[(bi * 128 + t // 16 + 16 * i, bj * 16 + t % 16)] += 1
    assert len(seen) == rows * (K // 8) and set(seen.values()) == {1}
    # k_int4_g128: CTA b -> group b // nb, channels (b % nb) * 128 + thread, those < N
    for N in (72, 4096, 200):
        nb = cdiv(N, 128)
        pairs = Counter()
        for b in range(nb * (K // 128)):
            g = b // nb
            for t in range(128):
                n = (b - g * nb) * 128 + t
                if n < N:
                    pairs[(g, n)] += 1
        assert len(pairs) == (K // 128) * N and set(pairs.values()) == {1}


def test_int4_tile_staging_covers_the_tile_and_reads_without_bank_conflicts():
    # k_int4_g128 copies: copy j of thread t -> row 8 j + t / 16, 16-byte column t % 16
    seen = Counter((8 * j + t // 16, t % 16) for t in range(128) for j in range(16))
    assert len(seen) == 128 * 16 and set(seen.values()) == {1}
    pitch = 272                                   # kInt4Pitch
    assert pitch % 16 == 0 and pitch >= 256
    # thread t then reads row t at t * pitch + 16 o; a 16-byte shared load is served a quarter
    # warp (8 lanes) at a time, and those 8 lanes must fall in 8 different groups of 4 banks
    for o in range(16):
        for q0 in range(0, 128, 8):
            groups = {((t * pitch + 16 * o) // 4 % 32) // 4 for t in range(q0, q0 + 8)}
            assert len(groups) == 8


def mma_scale_offset(row, j, chunks):
    """quant.cu, scale_row_base(row) + scale_col_part(j) in the QLIN_SCALE_MMA tiling."""
    rr = row & 127
    base = (((row >> 7) * chunks) << 9) + ((rr & 31) << 4) + ((rr >> 5) << 2)
    return base + (((j >> 2) << 9) + (j & 3))


@pytest.mark.parametrize("rows,nsc", [(1, 4), (333, 16), (256, 40)])
def test_mma_scale_tiling_is_a_bijection_onto_the_padded_buffer(rows, nsc):
    rows_pad = cdiv(rows, 128) * 128
    offs = [mma_scale_offset(r, j, nsc // 4) for r in range(rows_pad) for j in range(nsc)]
    assert sorted(offs) == list(range(rows_pad * nsc))


def pick_split_mma(tiles, groups):
    """gemm_w4a16.cu, pick_split_mma (M <= 16)."""
    cs = 1
    while cs < 8 and tiles * (cs + 1) <= 2 * SMS and groups >= 2 * (cs + 1):
        cs += 1
    return cs


def pick_split(tiles, groups):
    """gemm_w4a16.cu, pick_split (the tcgen05 kernel, M > 16): at most 4 ways."""
    cs = 1
    while cs < 4 and tiles * cs * 2 <= SMS and groups >= 2 * cs * 2:
        cs *= 2
    return cs


@pytest.mark.parametrize("M,K,N", [(1, 4096, 4096), (16, 4096, 12288), (16, 12288, 4096), (64, 4096, 4096),
                                   (64, 12288, 4096), (5, 256, 72), (24, 512, 136), (33, 128, 136), (70, 1024, 256),
                                   (64, 2048, 1024)])
def test_w4a16_split_k_partitions_groups_and_columns(M, K, N):
    groups = K // 128
    if M <= 16:
        tiles = cdiv(N, 128) * cdiv(M, 16)
        cs = pick_split_mma(tiles, groups)
        assert tiles * cs <= max(2 * SMS, tiles)        # about one wave of two CTAs per SM
    else:
        tiles = cdiv(N, 128) * cdiv(M, 64)             # 64-token tiles
        cs = pick_split(tiles, groups)
    assert 1 <= cs <= 8
    # rank r of the cluster takes groups [groups*r/cs, groups*(r+1)/cs): a partition, none empty
    parts = [(groups * r // cs, groups * (r + 1) // cs) for r in range(cs)]
    assert parts[0][0] == 0 and parts[-1][1] == groups
    assert all(a[1] == b[0] for a, b in zip(parts, parts[1:]))
    assert all(b - a >= (2 if cs > 1 else 1) for a, b in parts)
    # and sums output columns [128*r/cs, 128*(r+1)/cs) of the tile over the cluster
    cols = [(128 * r // cs, 128 * (r + 1) // cs) for r in range(cs)]
    assert cols[0][0] == 0 and cols[-1][1] == 128 and all(a[1] == b[0] for a, b in zip(cols, cols[1:]))


def rows_variant(K):
    """quant.cu, rowwise: the per-row kernel a row of K elements runs."""
    nv = K // 8
    if nv <= 128 * 8:
        return (128, cdiv(nv, 128))
    if nv <= 256 * 8:
        return (256, cdiv(nv, 256))
    return "long"


def test_row_quantizer_tests_reach_every_dispatched_variant():
    import test_gpu_quant
    reachable = {(128, v) for v in range(1, 9)} | {(256, v) for v in range(5, 9)} | {"long"}
    assert {rows_variant(K) for _, K in test_gpu_quant.SHAPES_ROW} == reachable
    for K in range(8, 20000, 8):
        v = rows_variant(K)
        if v != "long":
            assert v in reachable and v[0] * v[1] * 8 >= K      # the CTA's vectors cover the row


def test_w4a16_parity_cases_reach_every_cluster_size():
    """The W4A16 parity shapes run both warp-level kernels (M <= 8, tokens as
    the B operand; 8 < M <= 16) with every split-K cluster size they pick (1 to
    8) and the tcgen05 kernel with 1, 2 and 4."""
    import test_gpu_gemm
    shapes = []
    for mark in test_gpu_gemm.test_w4a16_gemm.pytestmark + test_gpu_gemm.test_w4a16_gemm_bias.pytestmark:
        if mark.name == "parametrize":
            shapes += list(mark.args[1])
    mma8 = {pick_split_mma(cdiv(N, 128) * cdiv(M, 16), K // 128) for M, K, N in shapes if M <= 8}
    mma16 = {pick_split_mma(cdiv(N, 128) * cdiv(M, 16), K // 128) for M, K, N in shapes if 8 < M <= 16}
    tc = {pick_split(cdiv(N, 128) * cdiv(M, 64), K // 128) for M, K, N in shapes if M > 16}
    assert mma8 == set(range(1, 9)) and mma16 == set(range(1, 9)) and tc == {1, 2, 4}
