"""Pins for the oracle's LRU slot cache (CPU only).

1. The hand trace in tests/golden/lru_hand_trace.json.
2. A second, independent formulation -- victims by argmin over
   (timestamp, slot) with no recency list -- on thousands of random query
   sequences.
3. The invariants the pages fix: map and slot_key stay a bijection; no query
   evicts its own hits; when the pool can hold all of a chunk's experts,
   later queries never evict an earlier query's slots (FreeToken PR
   #676, the author's reply); with record_stats off no statistic moves.
"""
import json
import os

import numpy as np
import pytest

from conftest import GOLDEN
from oracle.slot_cache import BAD_ID, CAPACITY, OK, SlotCache


def test_hand_trace():
    g = json.load(open(os.path.join(GOLDEN, "lru_hand_trace.json")))
    ini = g["initial"]
    c = SlotCache.from_state(g["S"], g["L"], g["E"], ini["slot_key"], ini["slot_ts"], ini["clock"])
    for st in g["steps"]:
        status, misses = c.ensure(st["query"])
        assert status == st["status"]
        assert [list(m) for m in misses] == st["misses"]
        assert c.slot_key.tolist() == st["slot_key"]
        assert c.slot_ts.tolist() == st["slot_ts"]
        assert c.clock == st["clock"]
    assert c.map.tolist() == g["final_map"]


class ArgminLRU:
    """Timestamp formulation: victim = argmin over non-hit slots of (ts, slot),
    where empty slots have ts 0 and occupied slots ts >= 1."""

    def __init__(self, S, L, E, slot_key, slot_ts, clock):
        self.S, self.L, self.E = S, L, E
        self.key = list(slot_key)
        self.ts = list(slot_ts)
        self.clock = clock

    def ensure(self, keys):
        q = [k for k in keys if k != -1]
        if not q:
            return OK, []
        if any(k < 0 or k >= self.L * self.E for k in q) or any(a >= b for a, b in zip(q, q[1:])):
            return BAD_ID, []
        where = {k: s for s, k in enumerate(self.key) if k >= 0}
        hit_slots = {where[k] for k in q if k in where}
        miss = [k for k in q if k not in where]
        free = [s for s in range(self.S) if s not in hit_slots]
        if len(miss) > len(free):
            return CAPACITY, []
        self.clock += 1
        out = []
        taken = set()
        for k in miss:
            v = min((s for s in free if s not in taken),
                    key=lambda s: (self.ts[s] if self.key[s] >= 0 else 0, s))
            taken.add(v)
            out.append((k, v, self.key[v]))
            self.key[v] = k
        for s in hit_slots | taken:
            self.ts[s] = self.clock
        return OK, out


def _random_state(g, S, L, E):
    n = int(g.integers(0, S + 1))
    key = [-1] * S
    ts = [0] * S
    slots = g.permutation(S)[:n]
    keys = g.choice(L * E, size=min(n, L * E), replace=False)
    stamps = g.permutation(len(keys)) + 1
    for s, k, t in zip(slots, keys, stamps):
        key[int(s)] = int(k)
        ts[int(s)] = int(t)
    return key, ts, len(keys)


def test_argmin_formulation_agrees_on_random_sequences():
    g = np.random.default_rng(1234)
    n_checked = 0
    for trial in range(2500):
        S = int(g.integers(1, 9))
        L = int(g.integers(1, 3))
        E = int(g.integers(1, 13))
        key, ts, clock = _random_state(g, S, L, E)
        a = SlotCache.from_state(S, L, E, key, ts, clock)
        b = ArgminLRU(S, L, E, key, ts, clock)
        for step in range(4):
            W = int(g.integers(1, 6))
            q = sorted(set(int(v) for v in g.integers(0, L * E, size=W)))
            if g.random() < 0.05 and len(q) > 1:
                q = q[::-1]                     # not ascending: bad id
            q = q + [-1] * int(g.integers(0, 3))
            sa, ma = a.ensure(q)
            sb, mb = b.ensure(q)
            assert sa == sb, (trial, step)
            assert [tuple(m) for m in ma] == mb
            assert a.slot_key.tolist() == b.key
            assert a.slot_ts.tolist() == [t if k >= 0 else t for t, k in zip(b.ts, b.key)]
            n_checked += 1
    assert n_checked == 10000


@pytest.mark.parametrize("seed", range(8))
def test_invariants(seed):
    g = np.random.default_rng(seed)
    S, L, E = 12, 3, 10
    key, ts, clock = _random_state(g, S, L, E)
    c = SlotCache.from_state(S, L, E, key, ts, clock)
    for _ in range(50):
        q = sorted(set(int(v) for v in g.integers(0, L * E, size=int(g.integers(1, 6)))))
        before_map = c.map.copy()
        status, misses = c.ensure(q, record_stats=False)
        # bijection between map and slot_key
        for s in range(S):
            if c.slot_key[s] >= 0:
                assert c.map[c.slot_key[s]] == s
        assert (c.map >= 0).sum() == (c.slot_key >= 0).sum()
        if status == OK:
            hit_slots = {int(before_map[k]) for k in q if before_map[k] >= 0}
            assert not hit_slots & {slot for _, slot, _ in misses}
            for k in q:
                assert c.map[k] >= 0
        assert c.hits == c.misses == c.evictions == 0
        assert not c.decode_freq.any()


@pytest.mark.parametrize("seed", range(6))
def test_earlier_queries_survive_when_layer_fits(seed):
    """One layer's distinct experts in queries of W: when D <= S no later
    query of the same chunk evicts a slot an earlier query hit or filled."""
    g = np.random.default_rng(100 + seed)
    S, L, E, W = 40, 2, 32, 4
    key, ts, clock = _random_state(g, S, L, E)
    c = SlotCache.from_state(S, L, E, key, ts, clock)
    layer = int(g.integers(0, L))
    D = int(g.integers(1, E + 1))
    experts = sorted(g.choice(E, size=D, replace=False).tolist())
    keys = [layer * E + e for e in experts]
    held = {}
    for q0 in range(0, len(keys), W):
        q = keys[q0:q0 + W]
        status, misses = c.ensure(q)
        assert status == OK
        for k in held:
            assert c.map[k] == held[k], "an earlier query's slot was evicted"
        for k in q:
            held[k] = int(c.map[k])
    assert len(set(held.values())) == D


def test_record_stats_counts():
    c = SlotCache(4, 1, 6)
    c.ensure([0, 1], record_stats=True)
    c.ensure([1, 2, 3], record_stats=True)
    c.ensure([4], record_stats=True)          # evicts key 0 (least recent)
    assert c.stats() == {"hits": 1, "misses": 5, "evictions": 1}
    assert c.decode_freq.tolist() == [1, 2, 1, 1, 1, 0]
    snap = (c.stats(), c.decode_freq.copy())
    c.ensure([0, 5], record_stats=False)       # demand admission: no stats
    assert c.stats() == snap[0] and (c.decode_freq == snap[1]).all()
    assert c.map[0] >= 0 and c.map[5] >= 0


def test_a_later_querys_resident_expert_can_be_evicted_but_touched_ones_cannot():
    """The pages protect what earlier queries touched (the author's reply on
    FreeToken PR #676: LRU takes those last), not what a later query will
    hit: with a full pool, query 1's misses evict the oldest slots, which
    may hold an expert of query 2.  Pinned by hand: 4 slots, query width 2,
    chunk experts {0, 1, 2, 3} of one layer; slots hold 3 (oldest), 9, 8,
    1.  Query {0, 1}: 1 hits, 0 misses and evicts the oldest non-hit slot,
    the one holding 3, which query {2, 3} then misses again."""
    c = SlotCache.from_state(4, 1, 16, np.array([3, 9, 8, 1]), np.array([1, 2, 3, 4]), 4)
    st, m1 = c.ensure([0, 1])
    assert st == OK and m1 == [(0, 0, 3)]
    st, m2 = c.ensure([2, 3])
    assert st == OK and m2 == [(2, 1, 9), (3, 2, 8)]
    assert c.map[1] == 3 and c.map[0] == 0          # touched by query 1: kept


@pytest.mark.parametrize("seed", range(200))
def test_touched_slots_survive_the_chunk_with_a_full_pool(seed):
    """Random full pools and chunks that fit: every expert a query touched
    (hit or filled) keeps its slot through the rest of the chunk; an expert
    that was a hit in its own query keeps the slot it had before."""
    rng = np.random.default_rng(seed)
    E, L = int(rng.integers(8, 60)), int(rng.integers(1, 4))
    S = int(rng.integers(4, min(L * E, 80) + 1))
    keys = rng.choice(L * E, size=S, replace=False)
    c = SlotCache.from_state(S, L, E, keys.astype(np.int32),
                             rng.permutation(S).astype(np.int64) + 1, S)
    before = c.map.copy()
    D = int(rng.integers(1, min(S, E) + 1))
    layer = int(rng.integers(0, L))
    chunk = np.sort(rng.choice(E, size=D, replace=False)) + layer * E
    width = int(rng.integers(1, 6))
    touched = {}
    hits = set()
    for q0 in range(0, D, width):
        q = chunk[q0:q0 + width]
        for key in q:
            if c.map[key] >= 0:
                hits.add(int(key))
        st, _ = c.ensure(q)
        assert st == OK
        for key in q:
            touched[int(key)] = int(c.map[key])
        for key, slot in touched.items():
            assert c.map[key] == slot
    for key in hits:
        assert c.map[key] == before[key]
