"""GPU parity of the LRFU policy with chunk pins, through the C ABI.

Bit-exact against the oracle: every miss list, the map, slots, timestamps,
the Q32.32 scores and the pins, on the hand traces and on random query
sequences with decay shifts 0 (LFU), 2 and 7, queries grouped into chunks
sharing a pin tag.  Then the whole slot path under LRFU: tables and pins
follow the oracle given the tag of the call, the output matches it, and the
slot path equals the streamed path byte for byte.
"""
import json
import os

import numpy as np
import pytest
import torch

from conftest import GOLDEN
from gpu_util import Workload, cuda, i32, lib, status
from offloaded_expert_slot_gb300 import oes
from offloaded_expert_slot_gb300.configs import C2, scaled
from oracle.layer import forward_slots
from oracle.slot_cache import SlotCache
from test_gpu_layer import Run, check_close, gpu_stream
from test_gpu_slot_cache import STATUS

pytestmark = pytest.mark.gpu


class Lrfu:
    def __init__(self, S, L, E, k):
        lib()
        self.S, self.L, self.E = S, L, E
        self.h = oes.slot_cache_create(S, L, E)
        oes.slot_cache_set_policy(self.h, oes.OES_POLICY_LRFU, k)
        self.miss, self.n_miss, self.status = i32(3 * oes.OES_QUERY_MAX, -9), i32(1, -9), status()

    def ensure(self, layer, experts, tag):
        n = len(experts)
        dev = cuda(np.asarray(experts, dtype=np.int32)) if n else 0
        self.status.zero_()
        oes.slot_cache_ensure_tagged(self.h, layer, dev, n, 0, tag, self.miss, self.n_miss,
                                     self.status)
        torch.cuda.synchronize()
        nm = int(self.n_miss.item())
        m = self.miss.cpu().numpy()[: 3 * nm].reshape(nm, 3)
        return int(self.status.item()), [tuple(int(v) for v in r) for r in m]

    def same_as(self, o: SlotCache):
        st = oes.slot_cache_read_state(self.h, self.S, self.L, self.E)
        crf, pin = oes.slot_cache_read_lrfu(self.h, self.S)
        assert np.array_equal(st["map"], o.map) and np.array_equal(st["slot_key"], o.slot_key)
        assert np.array_equal(st["slot_ts"], o.slot_ts) and st["clock"] == o.clock
        assert [int(v) for v in crf] == o.crf
        assert [int(v) for v in pin] == o.pin

    def close(self):
        oes.slot_cache_destroy(self.h)


@pytest.mark.parametrize("trace", ["frequency", "pinning"])
def test_hand_traces_on_gpu(trace):
    g = json.load(open(os.path.join(GOLDEN, "lrfu_hand_trace.json")))
    c = Lrfu(g["S"], g["L"], g["E"], g["k"])
    crf_want = []
    for step in g[trace]:
        st, m = c.ensure(0, step["q"], step["tag"])
        assert st == 0 and [list(x) for x in m] == step["misses"]
        crf, _pin = oes.slot_cache_read_lrfu(c.h, g["S"])
        assert [int(v) / 2 ** 32 for v in crf] == step["crf"]
    c.close()


@pytest.mark.parametrize("seed", range(9))
def test_random_sequences_with_chunks(seed):
    rng = np.random.default_rng(700 + seed)
    k = [0, 2, 7][seed % 3]
    S = int(rng.choice([3, 17, 300, 1100]))
    L = int(rng.integers(1, 4))
    E = int(rng.choice([8, 64, 512]))
    c = Lrfu(S, L, E, k)
    o = SlotCache(S, L, E)
    o.set_policy("lrfu", k)
    tag = 0
    for chunk in range(12):
        tag = tag + 1 if rng.random() < 0.8 else 0             # some queries untagged
        layer = int(rng.integers(0, L))
        D = int(rng.integers(0, min(S, E) + 1))
        experts = sorted(rng.choice(E, size=D, replace=False).tolist())
        width = int(rng.integers(1, oes.OES_QUERY_MAX + 1))
        for q0 in range(0, max(D, 1), width):
            q = experts[q0:q0 + width]
            st, m = c.ensure(layer, q, tag)
            ost, om = o.ensure([layer * E + e for e in q], tag=tag)
            assert st == STATUS[ost], (seed, chunk)
            assert m == [tuple(x) for x in om], (seed, chunk)
        c.same_as(o)
    c.close()


def test_slot_path_under_lrfu():
    lib()
    cfg = scaled(C2, name="lrfu_layer", T=64, k=6, E=256, H=128, I=64, S=280, L=2, prefill=280)
    w = Workload(cfg, gen_device="cpu")
    oes.slot_cache_set_policy(w.cache, oes.OES_POLICY_LRFU, 3)
    o = SlotCache.from_state(cfg.S, cfg.L, cfg.E, w.prefill["slot_key"], w.prefill["slot_ts"],
                             w.prefill["clock"])
    o.set_policy("lrfu", 3)
    pool = w.oracle_pool()
    B = oes.oes_tile_plan(cfg.T * cfg.k, cfg.E)
    r = Run(w)
    for call in (1, 2):                     # the handle's tags: 1, then 2
        oes.moe_layer_forward_slots(w.cache, w.src, w.pool, cfg.layer, r.desc, r.chunk, 1)
        torch.cuda.synchronize()
        assert int(r.status.item()) == 0
        ores = forward_slots(cfg, w.rin, w.source_row, o, pool, block=B, record_stats=True, tag=call)
        assert len(ores["queries"]) >= 2
        st = oes.slot_cache_read_state(w.cache, cfg.S, cfg.L, cfg.E)
        crf, pin = oes.slot_cache_read_lrfu(w.cache, cfg.S)
        assert np.array_equal(st["map"], o.map) and [int(v) for v in crf] == o.crf
        assert [int(v) for v in pin] == o.pin
        check_close(r.out, ores["out"], "bf16")
    s = gpu_stream(w)
    assert torch.equal(s.out.view(torch.int16), r.out.view(torch.int16))
    w.close()
