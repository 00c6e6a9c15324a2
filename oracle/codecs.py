"""Oracle: element codecs for the stored KV bytes.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

[Pools 15], "second mapping: the KV store": FP8 KV is kept as raw bytes
(``store_dtype = uint8``) and viewed as FP8 on read.  The pages fix neither
the FP8 flavour nor the rounding; the reading taken here is OCP FP8 E4M3
("e4m3fn": bias 7, no infinities, NaN = S.1111.111, largest finite 448),
round-to-nearest-even with saturation to +-448, on the value ``x / scale``
computed in float32.  bf16 is the upper half of an IEEE float32 rounded to
nearest-even.

Both codecs are written from those definitions: the E4M3 encoder enumerates
the finite codes and picks the nearest one.
"""
from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------- bf16 ---
def bf16_encode(x) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    rounded = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        rounded = rounded.copy()
        rounded[nan] = ((u[nan] >> np.uint64(16)).astype(np.uint16) | np.uint16(0x0040))
    return rounded


def bf16_decode(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


# ---------------------------------------------------------------- e4m3 ---
def e4m3_value(code: int) -> float:
    """Value of one E4M3 code (OCP FP8, e4m3fn)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** (1 - 7)
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_POS_CODES = np.arange(0, 0x7F)               # 0x00 .. 0x7E: all finite >= 0
_POS_VALUES = np.array([e4m3_value(c) for c in _POS_CODES])
E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    table = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def e4m3_encode_scalar(x: float) -> int:
    """Round ``x`` (already float32) to the nearest E4M3 code, ties to the
    even code, saturating finite overflow to +-448; NaN -> 0x7F."""
    x = float(x)
    if x != x:
        return 0x7F
    sign = 0x80 if (x < 0 or (x == 0 and np.signbit(x))) else 0
    a = abs(x)
    if a >= E4M3_MAX:
        return sign | 0x7E
    d = np.abs(_POS_VALUES - a)
    best = np.flatnonzero(d == d.min())
    if len(best) == 1:
        code = int(_POS_CODES[best[0]])
    else:  # a tie between two neighbours: the even code wins
        even = [int(_POS_CODES[i]) for i in best if (int(_POS_CODES[i]) & 1) == 0]
        code = even[0]
    return sign | code


_BF16_TABLE = []


def _bf16_table() -> np.ndarray:
    """``e4m3_encode_scalar`` of every bf16 value, indexed by its bit pattern."""
    if not _BF16_TABLE:
        vals = bf16_decode(np.arange(65536, dtype=np.uint32).astype(np.uint16))
        _BF16_TABLE.append(np.array([e4m3_encode_scalar(v) for v in vals], dtype=np.uint8))
    return _BF16_TABLE[0]


def e4m3_encode(x, scale: float = 1.0) -> np.ndarray:
    """float values -> E4M3 codes of ``float32(x / scale)``."""
    f = np.asarray(x, dtype=np.float32) / np.float32(scale)
    bits = bf16_encode(f)
    if f.size > 4096 and np.array_equal(bf16_decode(bits), f):
        # Every value is a bf16 value: look the scalar rule up by bit pattern.
        return _bf16_table()[bits]
    flat = f.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    # Encode the distinct values once (inputs are mostly bf16 values).
    uniq, inv = np.unique(flat, return_inverse=True)
    codes = np.array([e4m3_encode_scalar(v) for v in uniq], dtype=np.uint8)
    out[:] = codes[inv]
    return out.reshape(f.shape)
