"""Byte layouts of the packed NVFP4 operands, as the C header documents them.

Written independently from the header's text (not from the library's code):

* codes: row-major ``[rows][K/2]`` bytes; element ``2i`` of a row in the low
  nibble of byte ``i``, element ``2i+1`` in the high nibble.
* scales: a ``rows x C`` matrix of e4m3 bytes (C = K/16) stored in 512-byte
  tiles.  Rows form 128-row blocks ``rb = r // 128``; columns form 4-column
  groups ``cb = c // 4``.  Tile ``(rb, cb)`` starts at byte
  ``(rb * (C // 4) + cb) * 512``; inside it, entry ``(r, c)`` is at byte
  ``(r % 32) * 16 + ((r // 32) % 4) * 4 + (c % 4)``.  The buffer holds
  ``ceil(rows / 128)`` row blocks; rows past ``rows`` are padding.
"""
from __future__ import annotations

import numpy as np


def sf_padded_rows(rows: int) -> int:
    return ((rows + 127) // 128) * 128


def sf_nbytes(rows: int, K: int) -> int:
    return sf_padded_rows(rows) * (K // 16)


def sf_offset(r, c, C: int):
    """Byte offset of scale (row r, scale-column c) in a buffer with C scale
    columns per row (vectorised over integer arrays r, c)."""
    r = np.asarray(r, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    tile = (r // 128) * (C // 4) + (c // 4)
    return tile * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (c % 4)


def sf_swizzle(scales: np.ndarray, pad_value: int = 0) -> np.ndarray:
    """[rows][C] uint8 -> flat uint8 buffer in the tiled layout (padding rows
    filled with ``pad_value``)."""
    rows, C = scales.shape
    if C % 4:
        raise ValueError("scale columns must be a multiple of 4 (K % 64 == 0)")
    out = np.full(sf_padded_rows(rows) * C, pad_value, dtype=np.uint8)
    r, c = np.meshgrid(np.arange(rows), np.arange(C), indexing="ij")
    out[sf_offset(r, c, C)] = scales
    return out


def sf_unswizzle(buf: np.ndarray, rows: int, C: int) -> np.ndarray:
    """Inverse of :func:`sf_swizzle` (drops padding rows)."""
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    if buf.size < sf_padded_rows(rows) * C:
        raise ValueError("scale buffer too small")
    r, c = np.meshgrid(np.arange(rows), np.arange(C), indexing="ij")
    return buf[sf_offset(r, c, C)]


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """[rows][K] 4-bit codes -> [rows][K/2] bytes, even element in the low nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    if codes.shape[-1] % 2:
        raise ValueError("K must be even")
    lo = codes[..., 0::2] & 0xF
    hi = codes[..., 1::2] & 0xF
    return (lo | (hi << 4)).astype(np.uint8)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    """[rows][K/2] bytes -> [rows][K] 4-bit codes (inverse of pack_nibbles)."""
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out
