"""GPU parity: the LRU ensure and the miss-row copies against the oracle.

Bit-exact: every miss list, n_miss, map, slot_key, slot_ts, clock, the
counters and decode_freq, and the status word.  Copies: miss slots hold the
source rows byte for byte, every other slot is untouched (vLLM fork PR #51,
Tests: rows already resident keep their bytes).
"""
import json
import os

import numpy as np
import pytest
import torch

from conftest import GOLDEN
from gpu_util import Workload, cuda, f32, i32, lib, status
from offloaded_expert_slot_gb300 import oes
from offloaded_expert_slot_gb300.configs import C2, C5, scaled
from offloaded_expert_slot_gb300.inputs import pool_prefill, router_inputs
from oracle.distinct import distinct_experts
from oracle.router import route_topk
from oracle.slot_cache import SlotCache

pytestmark = pytest.mark.gpu


class GpuCache:
    def __init__(self, S, L, E):
        lib()
        self.S, self.L, self.E = S, L, E
        self.h = oes.slot_cache_create(S, L, E)
        self.miss = i32(3 * oes.OES_QUERY_MAX, -9)
        self.n_miss = i32(1, -9)
        self.status = status()

    def load(self, slot_key, slot_ts, clock):
        oes.slot_cache_load_state(self.h, slot_key, slot_ts, clock)

    def ensure(self, layer, experts, record_stats=False):
        n = len(experts)
        dev = cuda(np.asarray(experts, dtype=np.int32)) if n else None
        self.status.zero_()
        oes.slot_cache_ensure(self.h, layer, dev if n else 0, n, record_stats, self.miss, self.n_miss,
                              self.status)
        torch.cuda.synchronize()
        nm = int(self.n_miss.item())
        m = self.miss.cpu().numpy()[: 3 * nm].reshape(nm, 3)
        return int(self.status.item()), [tuple(int(v) for v in r) for r in m]

    def state(self):
        return oes.slot_cache_read_state(self.h, self.S, self.L, self.E)

    def close(self):
        oes.slot_cache_destroy(self.h)


STATUS = {0: 0, 1: oes.OES_DEV_CAPACITY, 2: oes.OES_DEV_BAD_ID}


def assert_same(g: GpuCache, o: SlotCache):
    st = g.state()
    assert np.array_equal(st["map"], o.map)
    assert np.array_equal(st["slot_key"], o.slot_key)
    assert np.array_equal(st["slot_ts"], o.slot_ts)
    assert st["clock"] == o.clock
    assert (st["hits"], st["misses"], st["evictions"]) == (o.hits, o.misses, o.evictions)
    assert np.array_equal(st["decode_freq"], o.decode_freq)


def test_hand_trace_on_gpu():
    g = json.load(open(os.path.join(GOLDEN, "lru_hand_trace.json")))
    ini = g["initial"]
    c = GpuCache(g["S"], g["L"], g["E"])
    c.load(ini["slot_key"], ini["slot_ts"], ini["clock"])
    for st in g["steps"]:
        s, m = c.ensure(0, st["query"])
        assert s == STATUS[st["status"]]
        assert [list(x) for x in m] == st["misses"]
        now = c.state()
        assert now["slot_key"].tolist() == st["slot_key"]
        assert now["slot_ts"].tolist() == st["slot_ts"]
        assert now["clock"] == st["clock"]
    assert c.state()["map"].tolist() == g["final_map"]
    c.close()


@pytest.mark.parametrize("seed", range(6))
def test_random_sequences_against_oracle(seed):
    g = np.random.default_rng(500 + seed)
    S = int(g.choice([1, 3, 8, 33, 257, 1100]))
    L = int(g.integers(1, 4))
    E = int(g.choice([4, 16, 200]))
    c = GpuCache(S, L, E)
    n = int(g.integers(0, min(S, L * E) + 1))
    key = np.full(S, -1, np.int32)
    ts = np.zeros(S, np.int64)
    slots = g.permutation(S)[:n]
    key[slots] = g.choice(L * E, size=n, replace=False)
    ts[slots] = g.permutation(n) + 1
    c.load(key, ts, n)
    o = SlotCache.from_state(S, L, E, key, ts, n)
    for step in range(25):
        layer = int(g.integers(0, L))
        w = int(g.integers(0, min(E, oes.OES_QUERY_MAX) + 1))
        q = sorted(g.choice(E, size=w, replace=False).tolist())
        if g.random() < 0.1 and len(q) > 1:
            q = q[::-1]                                     # not ascending
        if g.random() < 0.05:
            q = q + [E + 3]                                 # out of range
        q = q + [-1] * int(g.integers(0, 3))
        q = q[: oes.OES_QUERY_MAX]
        rs = bool(g.random() < 0.5)
        s, m = c.ensure(layer, q, record_stats=rs)
        os_, om = o.ensure([layer * E + e if e >= 0 and e < E else (-1 if e == -1 else 10 ** 9)
                            for e in q], record_stats=rs)
        assert s == STATUS[os_], (seed, step)
        assert m == [tuple(x) for x in om]
        assert_same(c, o)
    c.close()


def test_decode_width_queries_on_prefilled_pool():
    """The decode-width workload: 1100 slots shared by 2 layers, 800
    pre-filled; the chunk's distinct experts of layer 0 in queries of 128,
    no statistics recorded (a demand admission)."""
    cfg = C2
    st = pool_prefill(cfg)
    c = GpuCache(cfg.S, cfg.L, cfg.E)
    c.load(st["slot_key"], st["slot_ts"], st["clock"])
    o = SlotCache.from_state(cfg.S, cfg.L, cfg.E, st["slot_key"], st["slot_ts"], st["clock"])
    ids, _ = route_topk(router_inputs(cfg)["logits"], cfg.k)
    d, D = distinct_experts(ids, cfg.E)
    assert d.size == 320 and 150 < D < 320
    for q0 in range(0, d.size, 128):
        q = d[q0:q0 + 128].tolist()
        s, m = c.ensure(0, q)
        os_, om = o.ensure([e if e < 0 else e for e in q])
        assert s == 0 and m == [tuple(x) for x in om]
        assert_same(c, o)
    assert c.state()["hits"] == 0 and not c.state()["decode_freq"].any()
    c.close()


def test_wide_pool_many_queries_with_stats():
    """1650 slots (the long-prefill pool), 48 layers, four layers admitted in
    full (512 experts each, four queries per layer), with statistics."""
    cfg = C5
    c = GpuCache(cfg.S, cfg.L, cfg.E)
    o = SlotCache(cfg.S, cfg.L, cfg.E)
    g = np.random.default_rng(9)
    for layer in (0, 1, 2, 3, 0, 7):
        experts = sorted(g.choice(cfg.E, size=int(g.integers(300, 513)), replace=False).tolist())
        for q0 in range(0, len(experts), 128):
            q = experts[q0:q0 + 128]
            s, m = c.ensure(layer, q, record_stats=True)
            os_, om = o.ensure([layer * cfg.E + e for e in q], record_stats=True)
            assert s == 0 and m == [tuple(x) for x in om]
        assert_same(c, o)
    c.close()


def test_copy_misses_moves_exactly_the_miss_rows():
    cfg = scaled(C2, E=40, H=128, I=64, S=50, L=3, prefill=30, wfmt="bf16")
    w = Workload(cfg, gen_device="cpu")
    c_ref = SlotCache.from_state(cfg.S, cfg.L, cfg.E, w.prefill["slot_key"], w.prefill["slot_ts"],
                                 w.prefill["clock"])
    opool = w.oracle_pool()
    miss, n_miss, st = i32(3 * 128), i32(1), status()
    for layer, experts in [(0, list(range(0, 40, 3))), (2, list(range(5, 25))), (1, [0, 39])]:
        dev = cuda(np.array(experts, np.int32))
        oes.slot_cache_ensure(w.cache, layer, dev, len(experts), 0, miss, n_miss, st)
        oes.slot_cache_copy_misses(w.src, w.pool, cfg.S, miss, n_miss, len(experts), st)
        _, om = c_ref.ensure([layer * cfg.E + e for e in experts])
        for key, slot, _ in om:
            opool[slot] = w.source_row(key // cfg.E, key % cfg.E)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    pool = w.pool.cpu().numpy()
    for s in range(cfg.S):
        assert np.array_equal(pool[s], opool[s]), s
    w.close()


def test_copy_misses_large_rows_and_offsets_past_2gib():
    """Full-size bf16 rows (9 MiB) copied into slots whose byte offsets exceed
    2^31 (vLLM fork PR #51: a 32-bit offset overflows past 8192 rows x 4 MiB).
    Slots below the top six hold other layers' keys, so the six misses take
    the six empty slots at the top of a 2.8 GB pool."""
    L = 60
    cfg = scaled(C2, E=6, S=300, L=1, prefill=0)
    w = Workload(cfg, with_pool=False)
    pool = torch.zeros((cfg.S, cfg.row_bytes), dtype=torch.uint8, device="cuda")
    assert (cfg.S - 6) * cfg.row_bytes > 2 ** 31
    cache = oes.slot_cache_create(cfg.S, L, cfg.E)
    key = np.full(cfg.S, -1, np.int32)
    ts = np.zeros(cfg.S, np.int64)
    key[: cfg.S - 6] = np.arange(cfg.E, cfg.E + cfg.S - 6)      # keys of layers >= 1
    ts[: cfg.S - 6] = np.arange(1, cfg.S - 5)
    oes.slot_cache_load_state(cache, key, ts, cfg.S)
    src = oes.oes_expert_source_create([w.src_bufs[0]] * L, cfg.E, cfg.row_bytes)
    miss, n_miss, st = i32(3 * 128), i32(1), status()
    oes.slot_cache_ensure(cache, 0, cuda(np.arange(6, dtype=np.int32)), 6, 0, miss, n_miss, st)
    oes.slot_cache_copy_misses(src, pool, cfg.S, miss, n_miss, 6, st)
    torch.cuda.synchronize()
    m = miss.cpu().numpy()[:18].reshape(6, 3)
    assert int(st.item()) == 0 and int(n_miss.item()) == 6
    assert m[:, 1].tolist() == list(range(cfg.S - 6, cfg.S))
    for key_, slot, old in m:
        assert old == -1 and int(slot) * cfg.row_bytes >= 2 ** 31
        assert torch.equal(pool[int(slot)].cpu(), w.src_bufs[0][int(key_)])
    assert int(pool[: cfg.S - 6].count_nonzero().item()) == 0
    oes.oes_expert_source_destroy(src)
    oes.slot_cache_destroy(cache)
    w.close()


@pytest.mark.parametrize("policy", ["lru", "lrfu"])
def test_largest_pool(policy):
    """OES_MAX_SLOTS slots (the ensure kernel's 64 KB sort buffer, above the
    default 48 KB shared-memory limit) over 4 layers of 4096 experts, half
    pre-filled; random queries of up to 128 keys, bit-exact against the
    oracle under LRU and LRFU."""
    S, L, E = oes.OES_MAX_SLOTS, 4, 4096
    g = np.random.default_rng(8192)
    c = GpuCache(S, L, E)
    n = S // 2
    key = np.full(S, -1, np.int32)
    ts = np.zeros(S, np.int64)
    slots = g.permutation(S)[:n]
    key[slots] = g.choice(L * E, size=n, replace=False)
    ts[slots] = g.permutation(n) + 1
    c.load(key, ts, n)
    o = SlotCache.from_state(S, L, E, key, ts, n)
    if policy == "lrfu":
        oes.slot_cache_set_policy(c.h, oes.OES_POLICY_LRFU, 4)
        o.set_policy("lrfu", 4)
    for step in range(30):
        layer = int(g.integers(0, L))
        q = sorted(g.choice(E, size=int(g.integers(1, oes.OES_QUERY_MAX + 1)), replace=False).tolist())
        s, m = c.ensure(layer, q, record_stats=True)
        os_, om = o.ensure([layer * E + e for e in q], record_stats=True)
        assert s == STATUS[os_] and m == [tuple(x) for x in om], step
    assert_same(c, o)
    if policy == "lrfu":
        crf, pin = oes.slot_cache_read_lrfu(c.h, S)
        assert [int(v) for v in crf] == o.crf
    c.close()


@pytest.mark.parametrize("policy", ["lru", "lrfu"])
def test_reset_returns_the_created_state(policy):
    """slot_cache_reset, queued on the stream after queries that were not
    waited for, leaves every table byte as slot_cache_create does (the
    snapshot of a fresh handle with the same policy); the policy stays, and
    queries after it follow the oracle from an empty cache."""
    g = np.random.default_rng(910 + (policy == "lrfu"))
    S, L, E = 40, 2, 64
    c = GpuCache(S, L, E)
    fresh = oes.slot_cache_create(S, L, E)
    if policy == "lrfu":
        oes.slot_cache_set_policy(c.h, oes.OES_POLICY_LRFU, 3)
        oes.slot_cache_set_policy(fresh, oes.OES_POLICY_LRFU, 3)

    def queries(n):
        out = []
        for _ in range(n):
            w = int(g.integers(0, S + 1))
            out.append((int(g.integers(0, L)), sorted(g.choice(E, size=w, replace=False).tolist()),
                        bool(g.random() < 0.5)))
        return out

    keep = []
    for layer, q, rs in queries(6):                         # queued, not waited for
        dev = cuda(np.asarray(q, dtype=np.int32)) if q else 0
        keep.append(dev)
        oes.slot_cache_ensure(c.h, layer, dev, len(q), rs, c.miss, c.n_miss, c.status)
    oes.slot_cache_reset(c.h)
    nb = oes.slot_cache_state_bytes(c.h)
    a = torch.empty(nb, dtype=torch.uint8, device="cuda")
    b = torch.empty(nb, dtype=torch.uint8, device="cuda")
    oes.slot_cache_snapshot(c.h, a)
    oes.slot_cache_snapshot(fresh, b)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    st = c.state()
    assert (st["map"] == -1).all() and (st["slot_key"] == -1).all() and st["clock"] == 0
    o = SlotCache(S, L, E)
    if policy == "lrfu":
        o.set_policy("lrfu", 3)
    for layer, q, rs in queries(12):
        s_, m = c.ensure(layer, q, record_stats=rs)
        os_, om = o.ensure([layer * E + e for e in q], record_stats=rs)
        assert s_ == STATUS[os_] and m == [tuple(x) for x in om]
    assert_same(c, o)
    if policy == "lrfu":
        crf, pin = oes.slot_cache_read_lrfu(c.h, S)
        assert [int(v) for v in crf] == o.crf and [int(v) for v in pin] == o.pin
    oes.slot_cache_destroy(fresh)
    c.close()


def test_tiny_workload_queries_of_four_on_its_six_slot_pool():
    """The tiny workload's own cache traffic: its gate logits, routing and
    distinct experts computed on the GPU, then every query of 4 ensured and
    its misses copied on its 6-slot pool with 3 experts pre-resident, each
    step bit for bit against the oracle (tables, miss lists, pool rows).
    The 8 distinct experts exceed the 6 slots, so its layer forward is
    streamed (capacity reading: FreeToken PR #676, the author's reply);
    the queries themselves fit, and follow the oracle."""
    from offloaded_expert_slot_gb300.configs import C1
    from oracle.router import gate_logits
    cfg = C1
    w = Workload(cfg, gen_device="cpu")
    T, k, E, H, W = cfg.T, cfg.k, cfg.E, cfg.H, cfg.query_width
    R = T * k
    logits, ids, wts = f32(T * E), i32(R), f32(R)
    oes.moe_gate_logits(w.x, w.gate, T, H, E, logits)
    oes.moe_route_topk(logits, T, E, k, ids, wts)
    Lq = min(R, E)
    dist_d, dcnt = i32(Lq, -9), i32(1, -9)
    oes.moe_distinct_experts(ids, R, E, dist_d, dcnt)
    torch.cuda.synchronize()
    o_ids, _ = route_topk(gate_logits(w.rin["x"], w.rin["gate"]), k)
    o_dist, o_D = distinct_experts(o_ids, E)
    assert np.array_equal(ids.cpu().numpy().reshape(T, k), o_ids)
    assert np.array_equal(dist_d.cpu().numpy(), o_dist) and int(dcnt.item()) == o_D
    assert o_D > cfg.S                       # the layer itself is refused by the slot path
    o = SlotCache.from_state(cfg.S, cfg.L, E, w.prefill["slot_key"], w.prefill["slot_ts"],
                             w.prefill["clock"])
    opool = w.oracle_pool()
    miss, n_miss, st = i32(3 * 128), i32(1), status()
    for q0 in range(0, Lq, W):
        n = min(W, Lq - q0)
        oes.slot_cache_ensure(w.cache, cfg.layer, dist_d.data_ptr() + 4 * q0, n, 0, miss,
                              n_miss, st)
        oes.slot_cache_copy_misses(w.src, w.pool, cfg.S, miss, n_miss, n, st)
        torch.cuda.synchronize()
        s_, om = o.ensure([int(e) for e in o_dist[q0:q0 + n]])
        assert s_ == 0 and int(st.item()) == 0
        nm = int(n_miss.item())
        got = [tuple(int(v) for v in r) for r in miss.cpu().numpy()[:3 * nm].reshape(nm, 3)]
        assert got == [tuple(x) for x in om], q0
        for key, slot, _ in om:
            opool[slot] = w.source_row(key // E, key % E)
        now = oes.slot_cache_read_state(w.cache, cfg.S, cfg.L, E)
        assert np.array_equal(now["slot_key"], o.slot_key)
        assert np.array_equal(now["slot_ts"], o.slot_ts)
        assert np.array_equal(now["map"], o.map)
        assert now["clock"] == o.clock
        pool = w.pool.cpu().numpy()
        for s in range(cfg.S):
            assert np.array_equal(pool[s], opool[s]), (q0, s)
    w.close()
