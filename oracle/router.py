"""Router: top-k experts per token with softmax-renormalised weights.

Test infrastructure only.  The pages only say the chunk "routes"
(FreeToken PR #676, Problem and Solution); the workloads fix "softmax-
renormalised top-k".  Readings taken where the pages are silent:
  * top-k is chosen on the fp32 logits, larger first, ties to the lower
    expert id;
  * softmax over all E experts, keep the top k, divide by their sum -- which
    equals a softmax over the k selected logits -- computed in fp64 and
    stored as fp32;
  * bf16 logits are widened to fp32 (exact: bf16 is fp32's upper half) and
    routed the same way;
  * a NaN logit ranks as -inf (a logit that is not a number is no evidence
    for its expert): it is taken only after every finite logit, in id order
    with the -inf ones, and gets weight 0 beside a finite winner.
"""
from __future__ import annotations

import numpy as np

from .numerics import bf16_to_f64


def gate_logits(x_bits: np.ndarray, gate_bits: np.ndarray) -> np.ndarray:
    """Tiny workload only: logits = x @ gate, bf16 inputs, fp64 sums, fp32 result."""
    return (bf16_to_f64(x_bits) @ bf16_to_f64(gate_bits)).astype(np.float32)


def route_topk(logits: np.ndarray, k: int):
    """Returns ids [T, k] int32 (descending logit, ties to the lower id) and
    weights [T, k] fp32."""
    logits = np.asarray(logits, dtype=np.float32)
    logits = np.where(np.isnan(logits), np.float32(-np.inf), logits)
    T, E = logits.shape
    assert 1 <= k <= E
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
        ids[t] = order
        sel = np.array([float(logits[t, e]) for e in order], dtype=np.float64)
        ex = np.exp(sel - sel.max())
        w[t] = (ex / ex.sum()).astype(np.float32)
    return ids, w


def route_topk_bf16(logit_bits: np.ndarray, k: int):
    """route_topk on bf16 logits given as uint16 bit patterns [T, E]."""
    return route_topk(bf16_to_f64(logit_bits).astype(np.float32), k)
