"""Reference decoding of the FP8 packed layout for the tests (no GPU):
E4M3 codes decoded from the format's definition (OCP 8-bit E4M3: sign, 4
exponent bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 NaN),
and the dequantised weights bf16(fp32(code value * row scale))."""
from __future__ import annotations

import numpy as np

from tests.common import f32_to_bf16_bits


def e4m3_table() -> np.ndarray:
    codes = np.arange(256)
    sign = np.where(codes & 0x80, -1.0, 1.0)
    e, m = (codes >> 3) & 15, codes & 7
    v = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return (sign * v).astype(np.float32)


def nearest_e4m3(x: np.ndarray) -> np.ndarray:
    """Brute force over every finite code: the nearest E4M3 value to each x
    (fp32), an exact tie going to the even mantissa; beyond 448 the nearest
    finite value is +-448 (saturation)."""
    tab = e4m3_table().astype(np.float64)
    finite = np.isfinite(tab)
    vals = tab[finite]
    even = ((np.arange(256)[finite] & 1) == 0)
    x = np.asarray(x, dtype=np.float64).reshape(-1, 1)
    dist = np.abs(vals[None, :] - x)
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    # among tied candidates prefer an even mantissa (two distinct values tie
    # only at a midpoint, where exactly one of them has an even mantissa)
    pick = np.where((cand & even[None, :]).any(axis=1, keepdims=True), cand & even[None, :], cand)
    idx = np.argmax(pick, axis=1)
    return vals[idx].astype(np.float32)


def dequant_rows_bf16_bits(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """bf16 bits of float32(value(code) * scale) rounded to nearest even,
    codes [rows, cols] uint8, scales [rows] float32."""
    vals = e4m3_table()[codes]
    prod = (vals * scales.astype(np.float32)[:, None]).astype(np.float32)
    return f32_to_bf16_bits(prod)


def fp8_tensor(buf: np.ndarray, off: int, rows: int, cols: int):
    """(codes [rows, cols], scales [rows]) of one matrix tensor of the FP8 layout."""
    codes = buf[off:off + rows * cols].reshape(rows, cols)
    soff = off + (rows * cols + 15) // 16 * 16
    scales = buf[soff:soff + 4 * rows].view(np.float32)
    return codes, scales
