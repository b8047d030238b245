"""Pins for the oracle's LRFU policy (CPU only).

* Hand traces (tests/golden/lrfu_hand_trace.json): frequency beats recency
  where LRU would not, and a chunk's pinned slot survives its later query,
  which without the pin would evict what the chunk had just loaded
  (gdevenyi's review comment on FreeToken PR #676).
* k = 0 (no decay) is LFU: a brute-force LFU over reference counts makes the
  same choices on random query sequences.
* The decay: an idle slot's CRF after n queries is within n units of
  2^32 * (1 - 2^-k)^n.
* With pins, no query of a chunk that fits the pool evicts a slot an earlier
  query of the same chunk touched; without pins LRFU does so on some
  sequences.
"""
import json
import os

import numpy as np
import pytest

from conftest import GOLDEN
from oracle.slot_cache import CRF_SAT, OK, ONE, SlotCache

G = json.load(open(os.path.join(GOLDEN, "lrfu_hand_trace.json")))


def fresh(k):
    c = SlotCache(G["S"], G["L"], G["E"])
    c.set_policy("lrfu", k)
    return c


@pytest.mark.parametrize("trace", ["frequency", "pinning"])
def test_hand_traces(trace):
    c = fresh(G["k"])
    for step in G[trace]:
        st, misses = c.ensure(step["q"], tag=step["tag"])
        assert st == OK
        assert [list(m) for m in misses] == step["misses"], step
        assert [x / ONE for x in c.crf] == step["crf"], step
    if trace == "pinning":
        c = fresh(G["k"])
        for step in G[trace][:-1]:
            c.ensure(step["q"], tag=step["tag"])
        _st, misses = c.ensure(G[trace][-1]["q"], tag=0)
        assert [list(m) for m in misses] == G["unpinned_last_step_misses"]
    else:
        lru = SlotCache(G["S"], G["L"], G["E"])
        for step in G[trace][:-1]:
            lru.ensure(step["q"])
        _st, misses = lru.ensure(G[trace][-1]["q"])
        assert misses[0][2] == G["lru_would_evict_at_last_step"]


@pytest.mark.parametrize("seed", range(300))
def test_no_decay_is_lfu(seed):
    rng = np.random.default_rng(seed)
    S, L, E = int(rng.integers(2, 10)), int(rng.integers(1, 3)), int(rng.integers(3, 12))
    c = SlotCache(S, L, E)
    c.set_policy("lrfu", 0)
    count = {}                            # key -> references since it was loaded
    where = {}                            # key -> slot
    held = [None] * S
    for _ in range(int(rng.integers(1, 40))):
        n = int(rng.integers(1, min(S, L * E) + 1))
        q = sorted(rng.choice(L * E, size=n, replace=False).tolist())
        st, misses = c.ensure(q)
        assert st == OK
        hits = [x for x in q if x in where]
        for x in hits:
            count[x] += 1
        hit_slots = {where[x] for x in hits}
        order = sorted((s for s in range(S) if s not in hit_slots),
                       key=lambda s: (0 if held[s] is None else count[held[s]], s))
        want = []
        for x, s in zip([x for x in q if x not in where or where[x] is None], order):
            old = held[s]
            if old is not None:
                del where[old]
                del count[old]
            held[s], where[x], count[x] = x, s, 1
            want.append((x, s, -1 if old is None else old))
        assert misses == want
        assert [0 if h is None else count[h] * ONE for h in held] == c.crf


@pytest.mark.parametrize("k", [1, 2, 5, 9])
def test_decay_rate(k):
    c = SlotCache(4, 1, 8)
    c.set_policy("lrfu", k)
    c.ensure([0])                                  # slot 0 holds key 0 with CRF 1.0
    for n in range(1, 60):
        c.ensure([1 + (n % 3)])                    # other keys; key 0 is never hit
        if c.map[0] < 0:
            break
        want = ONE * (1 - 2.0 ** -k) ** n
        assert abs(c.crf[int(c.map[0])] - want) <= n + 1


@pytest.mark.parametrize("seed", range(200))
def test_pins_protect_a_chunks_earlier_queries(seed):
    rng = np.random.default_rng(1000 + seed)
    S, E = int(rng.integers(4, 20)), int(rng.integers(6, 30))
    k = int(rng.integers(0, 6))
    c = SlotCache(S, 1, E)
    c.set_policy("lrfu", k)
    for tag in range(1, 8):
        D = int(rng.integers(1, min(S, E) + 1))
        chunk = sorted(rng.choice(E, size=D, replace=False).tolist())
        width = int(rng.integers(1, 5))
        touched = {}
        for q0 in range(0, D, width):
            st, _m = c.ensure(chunk[q0:q0 + width], tag=tag)
            assert st == OK
            for x in chunk[q0:q0 + width]:
                touched[x] = int(c.map[x])
            for x, s in touched.items():
                assert c.map[x] == s


def test_without_pins_lrfu_evicts_an_earlier_querys_slot():
    found = 0
    for seed in range(200):
        rng = np.random.default_rng(5000 + seed)
        S, E = 6, 12
        c = SlotCache(S, 1, E)
        c.set_policy("lrfu", 2)
        for _ in range(20):                        # build up frequent keys
            c.ensure(sorted(rng.choice(4, size=2, replace=False).tolist()))
        chunk = sorted(rng.choice(range(4, E), size=S, replace=False).tolist())
        first = chunk[:3]
        c.ensure(first)
        c.ensure(chunk[3:])
        if any(c.map[x] < 0 for x in first):
            found += 1
    assert found > 0


def test_saturation():
    c = SlotCache(2, 1, 4)
    c.set_policy("lrfu", 0)
    c.crf = [CRF_SAT - 5, 0]
    c.slot_key[0] = 0
    c.map[0] = 0
    c.ensure([0])
    assert c.crf[0] == CRF_SAT
