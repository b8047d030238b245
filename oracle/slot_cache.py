"""LRU slot cache with an explicit recency list: the ensure step.

Test infrastructure only.  Sources:
  * FreeToken PR #676, Solution: the chunk's distinct experts reach the
    cache in queries of at most 128; a query's misses are copied before the
    following query may evict; a prefill's admissions change neither the
    decode-frequency counts nor the LRU statistics.
  * The author's reply on that page: LRU only; an earlier query's slots need
    no pin, since LRU takes them last and the pool is at least as large as
    the set of experts a layer routes to.
  * vLLM fork PR #48, What: one bank shared by all layers, keyed by
    (layer, expert).

The pool has S slots shared by L layers; key = layer * E + expert.

Readings taken where the pages are silent:
  * recency is an explicit list of slots, least recent first; empty slots
    start at the front in slot order;
  * one query is one tick of the clock; every slot a query touches (its hits
    and its fills) moves to the back in ascending slot order and gets the
    query's timestamp;
  * victims are the first slots of the list that the query does not hit;
    the i-th smallest missing key takes the i-th victim;
  * a query with more misses than non-hit slots changes nothing and reports
    a capacity error; a query that is not strictly ascending, or holds a key
    outside [0, L*E), changes nothing and reports a bad id; -1 entries are
    padding and ignored; a query with no valid key is a no-op;
  * with record_stats the counters hits, misses and evictions grow by the
    query's counts and decode_freq[key] grows by one for every key of the
    query; without it none of them changes, while recency still does.

LRFU (policy "lrfu"), the scored eviction the pages name (FreeToken PR
#676: one author's build admits by LRFU; gdevenyi's review comment there:
with a scored policy the earlier queries' slots of a chunk need pinning
against the later ones).  The pages give no formula; this is the published
LRFU (Lee et al., IEEE Trans. Computers 2001): each slot's combined recency
and frequency CRF(t) = F(0) + F(t - t_last) * CRF(t_last) with
F(x) = c^x, the victim being the smallest CRF.  Readings:
  * CRF is Q32.32 fixed point (1.0 = 2^32), saturating at 2^51 - 1;
  * one query is one tick: first every slot decays once,
    CRF -= CRF >> k (c = 1 - 2^-k; k = 0: no decay, LFU), then the victims
    are the non-hit, unpinned slots in ascending (CRF, slot) order, empty
    slots counting as 0; then each hit gains 1.0 and each fill starts at
    1.0;
  * a query with a tag t != 0 excludes the slots whose pin is t, and pins
    every slot it touches to t: the queries of one chunk share a tag, so a
    later query never evicts what an earlier one loaded or hit;
  * timestamps, the clock and the statistics move as under LRU.
"""
from __future__ import annotations

import numpy as np

OK = 0
CAPACITY = 1
BAD_ID = 2

ONE = 1 << 32                # CRF 1.0
CRF_SAT = (1 << 51) - 1


class SlotCache:
    def __init__(self, S: int, L: int, E: int):
        self.S, self.L, self.E = S, L, E
        self.map = np.full(L * E, -1, dtype=np.int32)
        self.slot_key = np.full(S, -1, dtype=np.int32)
        self.slot_ts = np.zeros(S, dtype=np.int64)
        self.recency = list(range(S))          # front = least recent
        self.clock = 0
        self.hits = 0
        self.misses = 0
        self.evictions = 0
        self.decode_freq = np.zeros(L * E, dtype=np.int64)
        self.policy, self.lrfu_k = "lru", 0
        self.crf = [0] * S                     # Q32.32, Python ints
        self.pin = [0] * S

    def set_policy(self, policy: str, k: int = 0):
        """LRFU scores start at 1.0 for every occupied slot; pins are cleared."""
        self.policy, self.lrfu_k = policy, int(k)
        self.crf = [ONE if self.slot_key[s] >= 0 else 0 for s in range(self.S)]
        self.pin = [0] * self.S

    @classmethod
    def from_state(cls, S, L, E, slot_key, slot_ts, clock):
        c = cls(S, L, E)
        c.slot_key = np.asarray(slot_key, dtype=np.int32).copy()
        c.slot_ts = np.asarray(slot_ts, dtype=np.int64).copy()
        c.clock = int(clock)
        for s in range(S):
            if c.slot_key[s] >= 0:
                c.map[c.slot_key[s]] = s
        empty = [s for s in range(S) if c.slot_key[s] < 0]
        full = sorted((s for s in range(S) if c.slot_key[s] >= 0),
                      key=lambda s: (int(c.slot_ts[s]), s))
        c.recency = empty + full
        c.crf = [ONE if c.slot_key[s] >= 0 else 0 for s in range(S)]
        return c

    def ensure(self, keys, record_stats: bool = False, tag: int = 0):
        """Admit one query.  Returns (status, misses) with misses a list of
        (key, slot, evicted_key or -1) in ascending key order.  tag: the
        chunk's pin tag (LRFU only; 0 = none)."""
        q = [int(v) for v in keys if int(v) != -1]
        if not q:
            return OK, []
        for i, v in enumerate(q):
            if v < 0 or v >= self.L * self.E or (i and q[i - 1] >= v):
                return BAD_ID, []
        hit_keys = [v for v in q if self.map[v] >= 0]
        miss_keys = [v for v in q if self.map[v] < 0]
        hit_slots = {int(self.map[v]) for v in hit_keys}
        lrfu = self.policy == "lrfu"
        if lrfu:
            k = self.lrfu_k
            decayed = [c - (c >> k) if k else c for c in self.crf]
            pinned = {s for s in range(self.S) if tag and self.pin[s] == tag}
            pool = [s for s in range(self.S) if s not in hit_slots and s not in pinned]
            score = lambda s: (0 if self.slot_key[s] < 0 else min(decayed[s], CRF_SAT), s)
            candidates = sorted(pool, key=score)
        else:
            candidates = [s for s in self.recency if s not in hit_slots]
        if len(miss_keys) > len(candidates):
            return CAPACITY, []
        victims = candidates[: len(miss_keys)]
        self.clock += 1
        if lrfu:
            self.crf = decayed
            for s in hit_slots:
                self.crf[s] = min(self.crf[s] + ONE, CRF_SAT)
            for s in victims:
                self.crf[s] = ONE
            if tag:
                for s in hit_slots | set(victims):
                    self.pin[s] = tag
        out = []
        for key, slot in zip(miss_keys, victims):
            old = int(self.slot_key[slot])
            if old >= 0:
                self.map[old] = -1
            self.map[key] = slot
            self.slot_key[slot] = key
            out.append((key, slot, old))
        touched = sorted(hit_slots | set(victims))
        touched_set = set(touched)
        self.recency = [s for s in self.recency if s not in touched_set] + touched
        for s in touched:
            self.slot_ts[s] = self.clock
        if record_stats:
            self.hits += len(hit_keys)
            self.misses += len(miss_keys)
            self.evictions += sum(1 for _, _, old in out if old >= 0)
            for v in q:
                self.decode_freq[v] += 1
        return OK, out

    def stats(self):
        return {"hits": self.hits, "misses": self.misses, "evictions": self.evictions}
