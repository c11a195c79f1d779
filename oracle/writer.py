"""The oracle of the cache writer: a record's rotary coordinates turned by its position, then
the record quantized to the cache's storage format (TEST INFRASTRUCTURE ONLY, like the rest
of this package).

Sources: the course's FP4 lesson ("How DeepSeek stores its main KV cache in four-bit
numbers": section 3, a code picks an E2M1 level and a scale shared by its group sets its
size; section 4, one E4M3 scale per 16 channels, quantization after RoPE, the local
sliding-window cache in FP8) and "DeepSeek-V4.1-Flash explained", section 7.

Readings (the pages do not describe the scale-selection kernel):
* FP4 group scale: the smallest E4M3 value at or above amax / 6 (6 = the largest E2M1
  level), so no element of the group clips; amax beyond 6 x 448 saturates at 448.
* each value x / scale rounds to the nearest E2M1 level, ties to the even code (the
  round-to-nearest-even of IEEE arithmetic; the lesson's teaching widget sends ties to the
  lower value and notes that hardware rounding can differ).
* FP8 rows: one fp32 scale amax / 448 per row (1 for an all-zero row), codes = E4M3 of
  x / scale, round to nearest even.
* RoPE on the last 64 coordinates by the record's position, pairs (448 + 2i, 449 + 2i),
  frequencies theta^(-2i/64), as for the query.

Every step that decides an integer code runs in float32, the kernel's precision: the
quotients x / scale and amax / 6 are IEEE float32 divisions, and the rotation forms
x cos - y sin and x sin + y cos from float32 products of float32 inputs with cos and sin
computed in float64 and rounded to float32.
"""
from __future__ import annotations

import numpy as np

from .csa2 import e4m3_to_f64, e2m1_to_f64

__all__ = ["e4m3_round", "e2m1_round", "bf16_round", "fp4_quantize", "fp8_quantize_rows", "rotate_f32",
           "write_records"]

# the 127 non-negative finite E4M3 values, in code order (0x00 .. 0x7E)
_E4M3 = e4m3_to_f64(np.arange(127, dtype=np.uint8))
# the 8 non-negative E2M1 magnitudes, in code order (0 .. 7)
_E2M1 = e2m1_to_f64(np.arange(8))


def _round_to_table(mag, table):
    """Index of the nearest table value to each magnitude (table ascending), ties to the even
    index (the even code); magnitudes beyond the table's end saturate at its last entry."""
    mag = np.asarray(mag, np.float64)
    hi = np.searchsorted(table, mag, side="left").clip(0, len(table) - 1)  # first >= mag
    lo = (hi - 1).clip(0, None)
    d_hi = table[hi] - mag
    d_lo = mag - table[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    idx = np.where(mag >= table[-1], len(table) - 1, np.where(pick_lo, lo, hi))
    return idx


def e4m3_round(x) -> np.ndarray:
    """E4M3 code of each float32 value: nearest finite value, ties to the even code,
    saturating at 448, the sign kept (also on zero) (OCP FP8 E4M3, with the
    round-to-nearest-even and saturation of a conversion to a format without infinities)."""
    x = np.asarray(x, np.float32).astype(np.float64)
    idx = _round_to_table(np.abs(x), _E4M3)
    return (idx | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)  # the sign survives a zero result


def bf16_round(x) -> np.ndarray:
    """bf16 bit patterns (uint16) of float32 values: the upper 16 bits after rounding the lower
    16 to nearest, ties to an even upper half (IEEE round-to-nearest-even into bf16's 8
    significant bits); finite inputs only."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def e2m1_round(q) -> np.ndarray:
    """E2M1 code (4 bits) of each value: nearest level, ties to the even code, saturating at 6."""
    q = np.asarray(q, np.float32).astype(np.float64)
    idx = _round_to_table(np.abs(q), _E2M1)
    return (idx | np.where(np.signbit(q), 0x8, 0)).astype(np.uint8)  # the sign survives a zero result


def fp4_quantize(x, group: int):
    """FP4 record(s) [..., D] float32 -> (codes [..., D/2] two per byte, low nibble the even
    channel; scale codes [..., D/group] E4M3)."""
    x = np.asarray(x, np.float32)
    lead, D = x.shape[:-1], x.shape[-1]
    xg = x.reshape(*lead, D // group, group)
    amax = np.abs(xg).max(-1)
    s = (amax / np.float32(6.0)).astype(np.float32)  # IEEE float32 division
    scode = np.searchsorted(_E4M3, s.astype(np.float64), side="left").clip(0, 126).astype(np.uint8)
    sval = _E4M3[scode].astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(sval[..., None] > 0, xg / sval[..., None], np.float32(0.0)).astype(np.float32)
    code = e2m1_round(q).reshape(*lead, D)
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).astype(np.uint8)
    return packed, scode


def fp8_quantize_rows(x):
    """FP8 row(s) [..., D] float32 -> (codes [..., D] E4M3, scale [...] float32)."""
    x = np.asarray(x, np.float32)
    amax = np.abs(x).max(-1)
    scale = np.where(amax > 0, (amax / np.float32(448.0)).astype(np.float32), np.float32(1.0)).astype(np.float32)
    q = (x / scale[..., None]).astype(np.float32)
    return e4m3_round(q), scale


def rotate_f32(x, pos, theta: float, R: int = 64):
    """RoPE of the last R coordinates of float32 record(s) [..., D] at positions pos [...]:
    pair i = (D-R+2i, D-R+2i+1) turns by pos * theta^(-2i/R); cos and sin in float64,
    rounded to float32; each product and sum in float32.  (The float64 cos and sin may
    differ from another implementation's in the last bit; the float32 values they round to
    then differ only when a value lies within 1e-16 relative of a float32 rounding
    boundary.)"""
    x = np.array(x, np.float32, copy=True)
    D = x.shape[-1]
    i = np.arange(R // 2, dtype=np.float64)
    inv = np.power(float(theta), -2.0 * i / R)
    a = np.asarray(pos, np.float64)[..., None] * inv
    c, s = np.cos(a).astype(np.float32), np.sin(a).astype(np.float32)
    xe = x[..., D - R::2].copy()
    xo = x[..., D - R + 1::2].copy()
    x[..., D - R::2] = (xe * c) - (xo * s)
    x[..., D - R + 1::2] = (xe * s) + (xo * c)
    return x


def write_records(x, pos, theta: float, fmt: str, group: int = 16):
    """The writer on records x [n, D] float32 at positions pos [n] (None: no rotation):
    fmt 'fp4' -> (codes [n, D/2], scale codes [n, D/group]); 'fp8' -> (codes [n, D], scales [n]);
    'bf16' -> (bf16 bit patterns [n, D], None)."""
    x = np.asarray(x, np.float32)
    if pos is not None:
        x = rotate_f32(x, pos, theta)
    if fmt == "fp4":
        return fp4_quantize(x, group)
    if fmt == "fp8":
        return fp8_quantize_rows(x)
    if fmt == "bf16":
        return bf16_round(x), None
    raise ValueError(fmt)
