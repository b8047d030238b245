"""Pins for the oracle's moe_align_block_size (CPU only)."""
import json
import os

import numpy as np
import pytest

from conftest import GOLDEN
from oracle.align import align_capacity, moe_align_block_size
from offloaded_expert_slot_gb300.inputs import uniform_routes


def test_hand_cases():
    for c in json.load(open(os.path.join(GOLDEN, "align_hand.json")))["cases"]:
        s, b, n, bad = moe_align_block_size(np.array(c["ids"]), c["E"], c["B"], c["ignore_invalid"])
        assert s.tolist() == c["sorted_ids"]
        assert b.tolist() == c["block_expert"]
        assert n == c["n_post_pad"]
        assert bad == c["bad"]


def check_align_invariants(ids, E, B, s, b, n):
    """Every valid route exactly once, inside a block of its own expert, in
    ascending route order; blocks padded with R; nothing past n_post_pad."""
    R = ids.size
    assert n % B == 0
    assert s.size == align_capacity(R, E, B)
    seen = np.zeros(R, dtype=np.int64)
    for pos in range(n):
        r = int(s[pos])
        e = int(b[pos // B])
        assert 0 <= e < E
        if r == R:
            continue
        assert ids[r] == e
        seen[r] += 1
    valid = (ids >= 0) & (ids < E)
    assert (seen[valid] == 1).all() and (seen[~valid] == 0).all()
    assert (s[n:] == R).all()
    assert (b[n // B:] == -1).all()
    blocks = b[: n // B]
    assert (np.diff(blocks) >= 0).all()            # experts ascending
    for e in np.unique(blocks):
        seg = s[:n][np.repeat(blocks == e, B)]
        real = seg[seg < R]
        assert (np.diff(real) > 0).all()
        assert (seg[: real.size] == real).all()    # padding only at the end
        assert seg.size == -(-real.size // B) * B


@pytest.mark.parametrize("seed", range(30))
def test_random_small_against_stable_sort(seed):
    """Brute force: the stable argsort of the expert ids (a library sort)
    gives the same route order once padding is removed."""
    g = np.random.default_rng(seed)
    E = int(g.integers(1, 20))
    R = int(g.integers(0, 65))
    B = int(g.choice([1, 2, 3, 4, 8, 16]))
    ids = g.integers(-1, E + 1, size=R)
    s, b, n, bad = moe_align_block_size(ids, E, B, ignore_invalid=False)
    check_align_invariants(ids, E, B, s, b, n)
    valid = (ids >= 0) & (ids < E)
    order = np.argsort(np.where(valid, ids, E + 10), kind="stable")[: int(valid.sum())]
    got = s[:n][s[:n] < R]
    assert got.tolist() == order.tolist()
    assert bad == bool((~valid).any())
    cnt = np.bincount(ids[valid], minlength=E)
    assert n == int(sum(-(-c // B) * B for c in cnt))


@pytest.mark.parametrize("E", [1023, 1024, 2100])
def test_past_1024_experts(E):
    """FreeToken PR #676, Tests: at 1023 and 2100 experts each route sits
    exactly once in a block of its own expert (smaller than the sweep's 8192 x 8 to keep
    the CPU suite short; the GPU tests run the full size)."""
    ids = uniform_routes(512, 8, E, seed=1006)
    s, b, n, _ = moe_align_block_size(ids, E, 64)
    check_align_invariants(ids, E, 64, s, b, n)


def test_capacity_bound():
    for R, E, B in [(0, 5, 4), (1, 1, 1), (10, 3, 8), (40960, 512, 128), (65536, 2100, 64)]:
        c = align_capacity(R, E, B)
        assert c % B == 0 and c >= R
        # worst case: min(E, R) experts each with a 1-route remainder
        assert c >= R + min(E, R) * (B - 1)
