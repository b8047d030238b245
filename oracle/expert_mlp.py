"""SwiGLU expert MLP over decoded expert rows, and the top-k combine.

Test infrastructure only.  The pages name the step (FreeToken PR #676,
Solution: the decode GEMM reused over the slot pool, each expert at its
slot) but not its formula; the workloads fix SwiGLU experts.  Readings:
  * an expert row holds w13 = [gate; up] stacked along the output axis
    (rows 0..I-1 gate, rows I..2I-1 up) and w2 [H, I];
  * y = w2 @ (silu(gate @ x) * (up @ x)), silu(g) = g / (1 + exp(-g));
  * NVFP4 weights decode exactly as e2m1 * e4m3 * global scale (vLLM fork
    PR #48 and FreeToken PR #676 use NVFP4 expert rows; the workload fixes
    "e2m1 values, e4m3 scale per 16 elements, fp32 per-tensor scale");
  * the combine is out[t] = sum over j = 0..k-1 of w[t, j] * y[t*k + j].
Everything is fp64; nothing is rounded to 16 bits in between.
"""
from __future__ import annotations

import numpy as np

from .numerics import bf16_to_f64, decode_e2m1_packed, decode_e4m3


def _nvfp4_sections(H: int, I: int):
    w13q = 0
    w13s = w13q + 2 * I * H // 2
    w2q = w13s + 2 * I * H // 16
    w2s = w2q + H * I // 2
    scal = w2s + H * I // 16
    return w13q, w13s, w2q, w2s, scal


def _decode_nvfp4_matrix(q: np.ndarray, s: np.ndarray, gs: float, rows: int, K: int):
    """q: [rows*K/2] bytes row-major; s: [K/64, rows, 4] e4m3 bytes; -> [rows, K]."""
    vals = decode_e2m1_packed(q.reshape(rows, K // 2), K)
    sc = decode_e4m3(s.reshape(K // 64, rows, 4).transpose(1, 0, 2).reshape(rows, K // 16))
    return vals * np.repeat(sc, 16, axis=1) * float(gs)


def expert_weights(row: np.ndarray, wfmt: str, H: int, I: int):
    """Decode one expert row to (w13 [2I, H], w2 [H, I]) in fp64."""
    row = np.asarray(row, dtype=np.uint8)
    if wfmt == "bf16":
        n13 = 2 * I * H
        w = row[: (n13 + H * I) * 2].view(np.uint16)
        return (bf16_to_f64(w[:n13]).reshape(2 * I, H),
                bf16_to_f64(w[n13:n13 + H * I]).reshape(H, I))
    if wfmt == "nvfp4":
        w13q, w13s, w2q, w2s, scal = _nvfp4_sections(H, I)
        gs13, gs2, _in13, _in2 = row[scal:scal + 16].view(np.float32)
        w13 = _decode_nvfp4_matrix(row[w13q:w13s], row[w13s:w2q], gs13, 2 * I, H)
        w2 = _decode_nvfp4_matrix(row[w2q:w2s], row[w2s:scal], gs2, H, I)
        return w13, w2
    raise ValueError(wfmt)


def input_scales(row: np.ndarray, H: int, I: int):
    """NVFP4 rows only: (w13 input scale, w2 input scale)."""
    *_, scal = _nvfp4_sections(H, I)
    s = np.asarray(row, dtype=np.uint8)[scal:scal + 16].view(np.float32)
    return float(s[2]), float(s[3])


def silu(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def swiglu_expert(x: np.ndarray, w13: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """x [n, H] fp64 -> y [n, H] fp64."""
    I = w2.shape[1]
    g = x @ w13[:I].T
    u = x @ w13[I:].T
    return (silu(g) * u) @ w2.T


def swiglu_expert_w4a4(x: np.ndarray, w13: np.ndarray, w2: np.ndarray, a13: float,
                       a2: float) -> np.ndarray:
    """W4A4: x [n, H] (bf16 values) quantised per 16 along H under a13, the
    SwiGLU output h quantised per 16 along I under a2 (its fp32 value decides
    the codes, as on the GPU), weights decoded as in W4A16.  fp64 otherwise."""
    from .quant import quantize_act
    I = w2.shape[1]
    xq = quantize_act(x.astype(np.float32), a13)[2] * a13
    h = silu(xq @ w13[:I].T) * (xq @ w13[I:].T)
    hq = quantize_act(h.astype(np.float32), a2)[2] * a2
    return hq @ w2.T


def combine(y: np.ndarray, w: np.ndarray, T: int, k: int) -> np.ndarray:
    """y [T*k, H], w [T, k] -> out [T, H]: sum over j in order 0..k-1."""
    H = y.shape[1]
    out = np.zeros((T, H), dtype=np.float64)
    for j in range(k):
        out += w[:, j:j + 1].astype(np.float64) * y[j::k]
    return out
