"""Number formats, decoded from their definitions (test infrastructure only).

bf16: the top 16 bits of an IEEE binary32.
e2m1 (4 bits, OCP MX / NVFP4 element): sign s, 2-bit exponent e (bias 1),
  1-bit mantissa m.  e == 0: value = m * 0.5 (subnormal); e > 0: value =
  2^(e-1) * (1 + m/2).  Magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
e4m3 (8 bits, "fn" variant, NVFP4 block scale): sign, 4-bit exponent (bias
  7), 3-bit mantissa.  e == 0: value = m/8 * 2^-6; e > 0: value =
  2^(e-7) * (1 + m/8); 0x7F / 0xFF are NaN (no infinities).
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round to nearest even bf16 via an exact fp32 intermediate where possible.

    Used only to express an fp64 result in the GPU's output precision for a
    report; comparisons are made in fp64.
    """
    f = np.asarray(a, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    return r.astype(np.uint16)


def e2m1_value(code: int) -> float:
    code = int(code) & 0xF
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    mag = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1.0 + m / 2.0)
    return -mag if s else mag


def e4m3_value(byte: int) -> float:
    byte = int(byte) & 0xFF
    s = (byte >> 7) & 1
    e = (byte >> 3) & 0xF
    m = byte & 7
    if e == 0xF and m == 7:
        return float("nan")
    mag = (m / 8.0) * 2.0 ** -6 if e == 0 else 2.0 ** (e - 7) * (1.0 + m / 8.0)
    return -mag if s else mag


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)


def decode_e2m1_packed(packed: np.ndarray, K: int) -> np.ndarray:
    """[rows, K/2] bytes, element 2i in the low nibble -> [rows, K] fp64."""
    p = np.asarray(packed, dtype=np.uint8)
    rows = p.shape[0]
    out = np.empty((rows, K), dtype=np.float64)
    out[:, 0::2] = E2M1_TABLE[p & 0xF]
    out[:, 1::2] = E2M1_TABLE[p >> 4]
    return out


def decode_e4m3(b: np.ndarray) -> np.ndarray:
    return E4M3_TABLE[np.asarray(b, dtype=np.uint8)]
