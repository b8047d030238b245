"""NVFP4 activation quantisation for the W4A4 expert GEMMs.

Test infrastructure only.  FreeToken PR #676, Solution and Tests: the W4A4
NVFP4 path quantises its activations under the maximum of the layer's input
scales (the layer's 2.0 / 3.0, never another slot's 9.0).  The pages fix the
format (e2m1 values with one e4m3 scale per 16 elements and a per-tensor fp32
scale) but not the rounding of each step; readings, all in fp32 as the kernel
computes them, with every rounding to nearest and ties to even:

  a      = max over the layer's experts of the input scale     (per GEMM)
  s      = amax(|v| over 16 consecutive K elements) / (6 * a)  (two fp32 ops)
  sf     = e4m3(s), saturating at 448; its value is exact in fp32
  q_i    = e2m1(v_i / (sf * a)), saturating at 6 (fp32 product and quotient);
           all zero when sf is 0
  value  = q_i * sf * a       (q_i * sf is exact in f16; a multiplies the sums)

Each code is chosen as the nearest representable value, ties to the even
code, by search over the format's table (its definition in numerics.py).
"""
from __future__ import annotations

import numpy as np

from .numerics import E2M1_TABLE, E4M3_TABLE

_E2M1_MAGS = E2M1_TABLE[:8]                        # codes 0..7: 0, 0.5, ..., 6
_E4M3_MAGS = E4M3_TABLE[:0x7F]                     # codes 0..0x7E: 0 .. 448 (0x7F is NaN)


def _nearest_even(mags: np.ndarray, x: np.ndarray) -> np.ndarray:
    """Code of the nearest magnitude to each x >= 0; ties to the even code."""
    x = np.asarray(x, dtype=np.float64)[..., None]
    d = np.abs(x - mags)
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    codes = np.arange(mags.size)
    # among tied candidates (at most two, adjacent), prefer the even code
    even = cand & (codes % 2 == 0)
    pick = np.where(even.any(axis=-1), np.argmax(even, axis=-1), np.argmax(cand, axis=-1))
    return pick.astype(np.uint8)


def e2m1_encode(x: np.ndarray) -> np.ndarray:
    """fp32 values -> e2m1 codes (sign bit 3), round to nearest even, saturating."""
    x = np.asarray(x, dtype=np.float32)
    mag = _nearest_even(_E2M1_MAGS, np.abs(x).astype(np.float64))
    return (mag | (np.signbit(x).astype(np.uint8) << 3)).astype(np.uint8)


def e4m3_encode_nonneg(x: np.ndarray) -> np.ndarray:
    """fp32 values >= 0 -> e4m3 codes, round to nearest even, saturating at 448."""
    return _nearest_even(_E4M3_MAGS, np.asarray(x, dtype=np.float32).astype(np.float64))


def quantize_act(v: np.ndarray, a: float):
    """v [..., K] (K a multiple of 16) -> (codes [..., K] e2m1, scales [..., K/16]
    e4m3, deq [..., K] fp64 = q * sf, without the factor a)."""
    v = np.asarray(v, dtype=np.float32)
    K = v.shape[-1]
    blk = v.reshape(*v.shape[:-1], K // 16, 16)
    a32 = np.float32(a)
    amax = np.abs(blk).max(axis=-1)
    s = amax / (np.float32(6.0) * a32)
    sc = e4m3_encode_nonneg(s)
    sf = E4M3_TABLE[sc].astype(np.float32)
    d = (sf * a32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(d > 0, blk / np.where(d > 0, d, np.float32(1)), np.float32(0)).astype(np.float32)
    q = e2m1_encode(r)
    deq = E2M1_TABLE[q] * sf.astype(np.float64)[..., None]
    return q.reshape(v.shape), sc, deq.reshape(v.shape)
