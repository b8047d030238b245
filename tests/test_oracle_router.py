"""Pins for the oracle's router and distinct-expert steps (CPU only)."""
import itertools
import json
import math
import os

import numpy as np
import pytest

from conftest import GOLDEN
from oracle.distinct import distinct_experts
from oracle.numerics import bf16_to_f64
from oracle.router import gate_logits, route_topk, route_topk_bf16


def test_router_hand_cases():
    cases = json.load(open(os.path.join(GOLDEN, "router_hand.json")))["cases"]
    for c in cases:
        ids, w = route_topk(np.array([c["logits"]], dtype=np.float32), c["k"])
        assert ids[0].tolist() == c["ids"]
        np.testing.assert_allclose(w[0], c["w"], rtol=1e-7, atol=0)


def test_router_bf16_logits_hand_case():
    """bf16 bit patterns with known values: 0x4000 = 2, 0x3f80 = 1, 0x3fc0 =
    1.5, 0x0000 = +0, 0x8000 = -0, 0xbf80 = -1, 0xc000 = -2, 0xff80 = -inf.
    Ordering by the raw (signed or unsigned) bits would put the negatives in
    the wrong place; -0 ties with +0 and the lower id wins."""
    bits = np.array([[0xbf80, 0x8000, 0x4000, 0x0000, 0xff80, 0x3fc0, 0xc000, 0x3f80]],
                    dtype=np.uint16)
    ids, w = route_topk_bf16(bits, 6)
    assert ids[0].tolist() == [2, 5, 7, 1, 3, 0]
    v = np.array([2.0, 1.5, 1.0, 0.0, 0.0, -1.0])
    want = np.exp(v - 2.0) / np.exp(v - 2.0).sum()
    np.testing.assert_allclose(w[0], want, rtol=1e-7, atol=0)
    ids, w = route_topk_bf16(bits, 8)
    assert ids[0].tolist() == [2, 5, 7, 1, 3, 0, 6, 4] and w[0, 7] == 0.0


@pytest.mark.parametrize("seed", range(20))
def test_router_brute_force_subsets(seed):
    """E=8, k=2 (the tiny workload's routing): the chosen set is the k-subset
    with the largest logits, ties resolved to the lexicographically smallest
    ids; weights equal the closed-form softmax over the chosen logits."""
    g = np.random.default_rng(seed)
    E, k = 8, 2
    # coarse values make ties frequent
    logits = (g.integers(-3, 4, size=(16, E)) * 0.5).astype(np.float32)
    ids, w = route_topk(logits, k)
    for t in range(logits.shape[0]):
        best = None
        for sub in itertools.combinations(range(E), k):
            vals = sorted((-float(logits[t, e]), e) for e in sub)
            if best is None or vals < best:
                best = vals
        want = [e for _, e in best]
        assert ids[t].tolist() == want
        z = [math.exp(float(logits[t, e])) for e in want]
        np.testing.assert_allclose(w[t], [v / sum(z) for v in z], rtol=2e-7)
        assert abs(float(w[t].astype(np.float64).sum()) - 1.0) < 1e-6


def test_router_full_topk_is_softmax():
    """k = E: the renormalised top-k is the plain softmax over all experts."""
    g = np.random.default_rng(3)
    logits = g.standard_normal((5, 6)).astype(np.float32)
    ids, w = route_topk(logits, 6)
    for t in range(5):
        p = np.exp(logits[t].astype(np.float64))
        p /= p.sum()
        np.testing.assert_allclose(w[t], p[ids[t]], rtol=2e-7)
        assert list(ids[t]) == sorted(range(6), key=lambda e: (-logits[t, e], e))


def test_gate_logits_is_bf16_matmul():
    """Gate logits: exact products of bf16 inputs; compared to numpy's fp64
    matmul (a library routine) of hand-widened values."""
    g = np.random.default_rng(5)
    xb = g.integers(0, 1 << 16, size=(4, 8), dtype=np.uint16) & 0x3FFF  # finite, modest
    gb = g.integers(0, 1 << 16, size=(8, 3), dtype=np.uint16) & 0xBFFF
    got = gate_logits(xb, gb)
    xf = np.array([[np.float32(np.uint32(int(v) << 16).view(np.float32)) for v in row] for row in xb],
                  dtype=np.float64)
    gf = np.array([[np.float32(np.uint32(int(v) << 16).view(np.float32)) for v in row] for row in gb],
                  dtype=np.float64)
    np.testing.assert_array_equal(got, np.matmul(xf, gf).astype(np.float32))
    assert bf16_to_f64(np.array([0x3F80], dtype=np.uint16))[0] == 1.0
    assert bf16_to_f64(np.array([0xC040], dtype=np.uint16))[0] == -3.0


@pytest.mark.parametrize("seed", range(10))
def test_distinct_brute_force(seed):
    g = np.random.default_rng(seed)
    E = int(g.integers(1, 40))
    R = int(g.integers(0, 60))
    ids = g.integers(-1, E, size=R).astype(np.int32)
    d, D = distinct_experts(ids, E)
    want = np.unique(ids[ids >= 0])
    assert D == want.size
    assert d.size == min(R, E)
    assert d[:D].tolist() == want.tolist()
    assert (d[D:] == -1).all()


def test_router_nan_ranks_as_minus_infinity():
    """A NaN logit ranks with the -inf ones: after every finite logit, ties to
    the lower id, weight 0 beside a finite winner."""
    nan, inf = np.float32(np.nan), np.float32(np.inf)
    logits = np.array([[0.5, nan, -inf, 1.0, nan, -2.0]], dtype=np.float32)
    ids, w = route_topk(logits, 5)
    assert ids.tolist() == [[3, 0, 5, 1, 2]]
    assert w[0, 3] == 0.0 and w[0, 4] == 0.0 and abs(float(w.sum()) - 1.0) < 1e-6
    # the same as writing -inf in their place
    ids2, w2 = route_topk(np.where(np.isnan(logits), -inf, logits), 5)
    assert np.array_equal(ids, ids2) and np.array_equal(w, w2)
