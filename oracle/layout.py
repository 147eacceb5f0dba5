"""The library's memory layouts, restated independently for the tests.

TEST INFRASTRUCTURE ONLY.  The oracle itself works on plain arrays: one code
per byte (outer x K) and a row-major scale matrix (outer x K/32).  The CUDA
library stores an MX tensor as

  * a data plane, outer x K, K contiguous: E4M3, E5M2 and int8 one code per
    byte; E2M1 and int4 two codes per byte, the element with even k in the
    low nibble; int2 four codes per byte, element k at bits 2*(k % 4);
  * a scale plane in the tensor-core scale-factor layout: the (padded)
    outer x K/32 scale matrix is cut into atoms of 128 rows x 4 scale columns
    (128 K elements); each atom is 512 contiguous bytes in which the scale of
    (row r, block j) sits at byte 16*(r % 32) + 4*((r % 128) // 32) + (j % 4);
    atoms follow each other K-chunk fastest:
    atom index = (r // 128) * ceil(K / 128) + j // 4.
    Padding rows and padding blocks hold code 0.

These helpers convert between the two, written from that description alone
(no code shared with the library), so that a test can compare the library's
bytes with the oracle's arrays and can build library-format inputs from
oracle-format codes.
"""
from __future__ import annotations

import numpy as np

ATOM_ROWS = 128
ATOM_BLOCKS = 4
ATOM_BYTES = 512


def scale_plane_bytes(outer: int, K: int) -> int:
    row_atoms = -(-outer // ATOM_ROWS)
    k_atoms = -(-K // (32 * ATOM_BLOCKS))
    return row_atoms * k_atoms * ATOM_BYTES


# bits per element code of each format (1 E4M3, 2 E2M1, 3 E5M2, 4 int8,
# 5 int4, 6 int2)
CODE_BITS = {1: 8, 2: 4, 3: 8, 4: 8, 5: 4, 6: 2}


def data_plane_bytes(fmt: int, outer: int, K: int) -> int:
    return outer * K * CODE_BITS[fmt] // 8


def _scale_offsets(outer: int, K: int) -> np.ndarray:
    """Byte offset of scale (r, j) in the tiled plane, shape outer x K/32."""
    nb = K // 32
    k_atoms = -(-K // (32 * ATOM_BLOCKS))
    r = np.arange(outer, dtype=np.int64)[:, None]
    j = np.arange(nb, dtype=np.int64)[None, :]
    atom = (r // ATOM_ROWS) * k_atoms + j // ATOM_BLOCKS
    inner = 16 * (r % 32) + 4 * ((r % ATOM_ROWS) // 32) + (j % ATOM_BLOCKS)
    return atom * ATOM_BYTES + inner


def tile_scales(scales: np.ndarray, K: int) -> np.ndarray:
    """Row-major outer x K/32 scale codes -> the library's tiled scale plane."""
    outer = scales.shape[0]
    out = np.zeros(scale_plane_bytes(outer, K), dtype=np.uint8)
    out[_scale_offsets(outer, K)] = scales
    return out


def untile_scales(tiled: np.ndarray, outer: int, K: int) -> np.ndarray:
    """The library's tiled scale plane -> row-major outer x K/32 codes."""
    tiled = np.asarray(tiled, dtype=np.uint8).reshape(-1)
    return tiled[_scale_offsets(outer, K)]


def pad_positions(outer: int, K: int) -> np.ndarray:
    """Boolean mask over the tiled plane: True where the byte is padding."""
    mask = np.ones(scale_plane_bytes(outer, K), dtype=bool)
    mask[_scale_offsets(outer, K).reshape(-1)] = False
    return mask


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """outer x K nibble codes -> outer x K/2 bytes, even k in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8) & 0xF
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def pack_codes(codes: np.ndarray, fmt: int) -> np.ndarray:
    """outer x K codes (one per byte) -> the library's data plane rows."""
    bits = CODE_BITS[fmt]
    c = np.asarray(codes, dtype=np.uint8)
    if bits == 8:
        return c.copy()
    if bits == 4:
        return pack_e2m1(c)
    c = c & 0x3
    return (c[:, 0::4] | (c[:, 1::4] << 2) | (c[:, 2::4] << 4) |
            (c[:, 3::4] << 6)).astype(np.uint8)


def unpack_codes(packed: np.ndarray, fmt: int, K: int) -> np.ndarray:
    """The library's data plane rows -> outer x K codes (one per byte)."""
    bits = CODE_BITS[fmt]
    p = np.asarray(packed, dtype=np.uint8)
    p = p.reshape(p.shape[0] if p.ndim > 1 else -1, K * bits // 8)
    if bits == 8:
        return p.copy()
    if bits == 4:
        return unpack_e2m1(p)
    out = np.empty((p.shape[0], K), dtype=np.uint8)
    for i in range(4):
        out[:, i::4] = (p >> (2 * i)) & 0x3
    return out


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """outer x K/2 bytes -> outer x K nibble codes."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty((p.shape[0], p.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = p & 0xF
    out[:, 1::2] = p >> 4
    return out
