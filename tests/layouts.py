"""Host-side reader for the tensor-core scale tiling (QLIN_SCALE_MMA).

Written from the layout stated in include/qlin.h, independently of the
kernels that produce it: 512-byte chunks of 128 rows x 4 scales, ordered
[row_tile][k_chunk], the scale of tile row r and chunk position j at byte
16*(r % 32) + 4*(r / 32) + j.
"""
import numpy as np


def mma_to_canonical(buf: np.ndarray, rows: int, n_scales: int) -> np.ndarray:
    """Flat uint8 buffer in the MMA tiling -> canonical [rows, n_scales]."""
    assert n_scales % 4 == 0
    tiles = (rows + 127) // 128
    chunks = n_scales // 4
    a = np.asarray(buf, np.uint8).reshape(-1)[: tiles * chunks * 512].reshape(tiles, chunks, 32, 4, 4)
    # a[tile, chunk, r % 32, r // 32, j]  ->  canonical[tile*128 + r, chunk*4 + j]
    c = a.transpose(0, 3, 2, 1, 4).reshape(tiles * 128, chunks * 4)
    return c[:rows]


def mma_padding_rows(buf: np.ndarray, rows: int, n_scales: int) -> np.ndarray:
    """The scale entries of the padding rows (rows .. next multiple of 128)."""
    tiles = (rows + 127) // 128
    chunks = n_scales // 4
    a = np.asarray(buf, np.uint8).reshape(-1)[: tiles * chunks * 512].reshape(tiles, chunks, 32, 4, 4)
    full = a.transpose(0, 3, 2, 1, 4).reshape(tiles * 128, chunks * 4)
    return full[rows:]
