"""Test-side packers: integer codes -> the packed byte layouts.

Written for the tests from the layout statement (int8 one byte per code; int4
and e2m1 two codes per byte with the even input in the low nibble -- the same
for the per-row and grouped variants and for ue8m0-scaled MXFP4; int3-g64
plane A [O][I/4] with four 2-bit fields per byte, then plane B [O][I/8] with
eight 1-bit fields per byte, least significant first).  The pins use them to
build matrices whose codes are known without the oracle's decoder, so a
decoding mistake in the oracle shows up as a mismatch.
"""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

INT8_ROW, INT4_ROW, INT4_G, INT3_G64, MXFP4_G32, MXFP4_E8M0, INT8_G = 1, 2, 4, 5, 7, 8, 13
BASE_FMTS = (INT8_ROW, INT4_G, INT3_G64, MXFP4_G32)
ALL_FMTS = BASE_FMTS + (INT4_ROW, INT8_G, MXFP4_E8M0)


def pack(fmt: int, codes: np.ndarray) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.int64)
    O, I = codes.shape
    if fmt in (INT8_ROW, INT8_G):
        return codes.astype(np.int8).view(np.uint8).reshape(-1).copy()
    if fmt in (INT4_G, INT4_ROW, MXFP4_G32, MXFP4_E8M0):
        c = codes.reshape(O, I // 2, 2)
        return ((c[..., 0] & 15) | ((c[..., 1] & 15) << 4)).astype(np.uint8).reshape(-1)
    if fmt == INT3_G64:
        lo = codes & 3
        hi = (codes >> 2) & 1
        a = lo.reshape(O, I // 4, 4)
        A = a[..., 0] | (a[..., 1] << 2) | (a[..., 2] << 4) | (a[..., 3] << 6)
        b = hi.reshape(O, I // 8, 8)
        B = np.zeros((O, I // 8), dtype=np.int64)
        for j in range(8):
            B |= b[..., j] << j
        return np.concatenate([A.astype(np.uint8).reshape(-1), B.astype(np.uint8).reshape(-1)])
    raise ValueError(fmt)


def random_codes(fmt: int, O: int, I: int, rng: np.random.Generator) -> np.ndarray:
    if fmt in (INT8_ROW, INT8_G):
        return rng.integers(-128, 128, size=(O, I))
    if fmt == INT3_G64:
        return rng.integers(0, 8, size=(O, I))
    return rng.integers(0, 16, size=(O, I))


def load_table(name: str):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


def e2m1_table() -> dict:
    return {int(c, 16): float(v) for c, v in load_table("e2m1_codes.txt")}


def values_of(fmt: int, codes: np.ndarray) -> np.ndarray:
    """Code -> value, from the golden e2m1 table and the stated offsets."""
    codes = np.asarray(codes, dtype=np.int64)
    if fmt in (INT8_ROW, INT8_G):
        return codes.astype(np.float64)
    if fmt in (INT4_G, INT4_ROW):
        return (codes - 8).astype(np.float64)
    if fmt == INT3_G64:
        return (codes - 4).astype(np.float64)
    tab = e2m1_table()
    lut = np.array([tab[c] for c in range(16)], dtype=np.float64)
    return lut[codes]


def group_of(fmt: int, I: int, gs: int | None = None) -> int:
    if fmt in (INT8_ROW, INT4_ROW):
        return I
    if fmt == INT3_G64:
        return 64
    if fmt in (MXFP4_G32, MXFP4_E8M0):
        return 32
    return gs or 32


def scale_values(fmt: int, scales: np.ndarray) -> np.ndarray:
    """Stored scales -> f64 values: f32 as is; ue8m0 bytes as 2^(e - 127) (OCP microscaling,
    255 = NaN)."""
    if fmt == MXFP4_E8M0:
        e = np.asarray(scales, dtype=np.int64)
        v = np.ldexp(1.0, e - 127)
        return np.where(e == 255, np.nan, v)
    return np.asarray(scales, dtype=np.float64)


def to_stored_scales(fmt: int, values: np.ndarray) -> np.ndarray:
    """f32 scale values -> the stored form: ue8m0 bytes hold the nearest power of two."""
    v = np.asarray(values, dtype=np.float64)
    if fmt == MXFP4_E8M0:
        e = 127 + np.round(np.log2(np.maximum(v, 2.0 ** -127)))
        return np.clip(e, 0, 254).astype(np.uint8)
    return v.astype(np.float32)


def draw_scales(fmt: int, n: int, rng: np.random.Generator, mu: float = -4.0, sigma: float = 0.5):
    return to_stored_scales(fmt, rng.lognormal(mu, sigma, size=n))


def dense(fmt: int, codes: np.ndarray, scales: np.ndarray, gs: int) -> np.ndarray:
    """Dense f64 matrix value(code) * scale[o][i // gs]."""
    O, I = codes.shape
    sc = scale_values(fmt, scales).reshape(O, I // gs)
    return values_of(fmt, codes) * np.repeat(sc, gs, axis=1)
