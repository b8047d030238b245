"""A complete check of W4A4 activation codes computed on the GPU from fp32
sums, against the oracle's fp64 values (test helper, CPU only).

FreeToken PR #676, Solution: the W4A4 path quantises the SwiGLU output h
per 16 along I under the max of the layer's input scales.  The GPU decides
each block's e4m3 scale and each e2m1 code from its own fp32 h, whose sums
run in another order than the oracle's fp64 ones.  So a code may differ from
the oracle's only where the oracle's value lies so close to a rounding
boundary that fp32 summation could put the GPU's value on the other side.
This module bounds that distance for every element and checks every code:

  * |h_gpu - h| <= dh, with dh from the fp32 accumulation of K exact
    products (f16 x f16 products are exact in fp32).  The tensor core adds
    16 products per instruction (kind::f16) and then adds that into the
    fp32 accumulator, K / 16 times; a split K range adds its two halves
    once more.  Counting every addition as one rounding of at most one ulp
    of a partial sum no larger than sum |x_k w_k|, in any order inside the
    instruction, bounds the error by (K/16 + 16 + 2) * 2^-23 * sum |x_k w_k|.
    Two roundings of the scale factors, and the SiLU and product, add
    2^-20 relative; the difference is carried through h = silu(g) u with
    max |silu'| <= 1.1;
  * the block's scale: amax(|h_gpu|) lies in [max(|h| - dh), max(|h| + dh)],
    so its e4m3 code lies between the codes of the two ends;
  * under that scale, each code lies between the e2m1 codes of
    (h - dh) / (sf a) and (h + dh) / (sf a).

Where the interval holds a single code (nearly always) the GPU's code must
be that code; where it straddles a boundary the GPU may take either side:
exactly one step at that boundary.
"""
from __future__ import annotations

import numpy as np

from oracle.numerics import E2M1_TABLE, E4M3_TABLE
from oracle.quant import e2m1_encode, e4m3_encode_nonneg, quantize_act

U = 2.0 ** -24
SILU_DMAX = 1.1          # max over x of |d/dx x sigmoid(x)| is 1.0998...


def h_with_bound(xq: np.ndarray, w13: np.ndarray, I: int):
    """xq [n, K] (activation codes times scale, fp64), w13 [2I, K] decoded
    weights: returns the oracle's fp64 h [n, I] and the bound dh [n, I]."""
    K = xq.shape[-1]
    adds = K // 16 + 16 + 2
    g = xq @ w13[:I].T
    u = xq @ w13[I:].T
    ax = np.abs(xq)
    sg = ax @ np.abs(w13[:I]).T
    su = ax @ np.abs(w13[I:]).T
    dg = adds * 2 * U * sg + 4 * U * np.abs(g)
    du = adds * 2 * U * su + 4 * U * np.abs(u)
    silu = g / (1.0 + np.exp(-g))
    h = silu * u
    dh = SILU_DMAX * dg * (np.abs(u) + du) + np.abs(silu) * du + 16 * U * np.abs(h) + 1e-30
    return h, dh


def _f32_down(x):
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)
    return np.where(f.astype(np.float64) > x, np.nextafter(f, np.float32(-np.inf)), f)


def _f32_up(x):
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)
    return np.where(f.astype(np.float64) < x, np.nextafter(f, np.float32(np.inf)), f)


def _block_fits(g, h, dh, a, sf):
    """Do the GPU's values g [16] fit the scale sf, code by code?"""
    if sf == 0.0:
        return bool((g == 0).all())
    d = float(np.float32(sf) * np.float32(a))
    lo = (h - dh) / d
    hi = (h + dh) / d
    lo = lo - np.abs(lo) * 4 * U - 1e-30          # the GPU's fp32 quotient
    hi = hi + np.abs(hi) * 4 * U + 1e-30
    v_lo = E2M1_TABLE[e2m1_encode(_f32_down(lo))]
    v_hi = E2M1_TABLE[e2m1_encode(_f32_up(hi))]
    q = g / sf
    on_grid = np.isin(np.abs(q), E2M1_TABLE[:8])
    return bool((on_grid & (q >= v_lo) & (q <= v_hi)).all())


def check_codes(g: np.ndarray, h: np.ndarray, dh: np.ndarray, a: float):
    """g: the GPU's q * sf values [n, K] (exact f16 values as fp64); h, dh:
    the oracle's fp64 values and their bounds.  Returns (bad_blocks,
    differing_codes, total_codes): bad_blocks lists (row, block) pairs no
    admissible scale and codes explain."""
    n, K = g.shape
    want = quantize_act(h.astype(np.float32), a)[2]
    gb = g.reshape(n, K // 16, 16)
    wb = want.reshape(n, K // 16, 16)
    hb = h.reshape(n, K // 16, 16)
    db = dh.reshape(n, K // 16, 16)
    differ = int((gb != wb).sum())
    bad = []
    d6 = np.float32(6.0) * np.float32(a)
    for r, b in zip(*np.nonzero((gb != wb).any(axis=-1))):
        hh, dd, gg = hb[r, b], db[r, b], gb[r, b]
        amax_lo = np.maximum(np.abs(hh) - dd, 0.0).max()
        amax_hi = (np.abs(hh) + dd).max()
        s_lo = _f32_down(amax_lo) / d6
        s_hi = _f32_up(amax_hi) / d6
        c_lo = int(e4m3_encode_nonneg(np.array([_f32_down(s_lo * (1 - 2 * U))]))[0])
        c_hi = int(e4m3_encode_nonneg(np.array([_f32_up(s_hi * (1 + 2 * U))]))[0])
        if not any(_block_fits(gg, hh, dd, a, E4M3_TABLE[c]) for c in range(c_lo, c_hi + 1)):
            bad.append((int(r), int(b)))
    return bad, differ, g.size
