"""Pins for the oracle's whole layer (CPU only).

* Closed form: experts that differ only by a power-of-two factor 2^e on w2
  give out[t] = (sum_j w[t, j] * 2^ids[t, j]) * MLP(x[t]); a route sent to
  the wrong expert, the wrong token or the wrong weight breaks it.
* The slot path equals the streamed path (FreeToken PR #676, Solution).
* 160 distinct experts go in as two queries (128, then 32), the copies of
  each landing before the next, with no statistic recorded (FreeToken PR
  #676, Tests).
* Resident rows the chunk does not evict are untouched (vLLM fork PR #51,
  Tests: rows already resident keep their bytes).
"""
import numpy as np
import pytest

from oracle.expert_mlp import swiglu_expert
from oracle.layer import forward_slots, forward_stream
from oracle.numerics import bf16_to_f64
from oracle.router import route_topk
from oracle.slot_cache import SlotCache
from offloaded_expert_slot_gb300.configs import C1, C4, scaled
from offloaded_expert_slot_gb300.inputs import (empty_slot_row, expert_layer_rows, f32_to_bf16_bits,
                                                pool_prefill, router_inputs)


def _bf16_row(w13, w2):
    return np.concatenate([f32_to_bf16_bits(w13).reshape(-1),
                           f32_to_bf16_bits(w2).reshape(-1)]).view(np.uint8)


def test_power_of_two_experts_closed_form():
    cfg = scaled(C1, T=12, k=3, E=6, H=16, I=8, logits="normal", S=6, prefill=0)
    g = np.random.default_rng(7)
    w13 = f32_to_bf16_bits(g.standard_normal((2 * cfg.I, cfg.H)).astype(np.float32) * 0.3)
    w2 = f32_to_bf16_bits(g.standard_normal((cfg.H, cfg.I)).astype(np.float32) * 0.3)
    w13f = bf16_to_f64(w13)
    w2f = bf16_to_f64(w2)
    rows = np.stack([_bf16_row(w13f.astype(np.float32), (w2f * 2.0 ** e).astype(np.float32))
                     for e in range(cfg.E)])
    rin = router_inputs(cfg)
    res = forward_stream(cfg, rin, lambda e: rows[e], block=4)
    ids, w = route_topk(rin["logits"], cfg.k)
    base = swiglu_expert(bf16_to_f64(rin["x"]), w13f, w2f)
    factor = (w.astype(np.float64) * np.exp2(ids)).sum(axis=1)
    np.testing.assert_allclose(res["out"], factor[:, None] * base, rtol=1e-12, atol=1e-14)


def _slot_setup(cfg):
    src = [expert_layer_rows(cfg, l).numpy() for l in range(cfg.L)]
    st = pool_prefill(cfg)
    cache = SlotCache.from_state(cfg.S, cfg.L, cfg.E, st["slot_key"], st["slot_ts"], st["clock"])
    empty = empty_slot_row(cfg)
    pool = {}
    for s in range(cfg.S):
        k = int(st["slot_key"][s])
        pool[s] = src[k // cfg.E][k % cfg.E] if k >= 0 else empty
    return src, cache, pool


def test_tiny_workload_is_refused_by_the_slot_path():
    """The tiny workload routes 16 tokens x top-2 over 8 experts into a 6-slot
    pool: min(R, E) = 8 > 6, so the slot path refuses it (it streams)."""
    src, cache, pool = _slot_setup(C1)
    res = forward_slots(C1, router_inputs(C1), lambda l, e: src[l][e], cache, pool, block=16)
    assert res["capacity"] and not res["ok"]


@pytest.mark.parametrize("cfg", [
    scaled(C1, S=8),
    scaled(C1, T=24, k=3, E=12, H=64, I=64, S=20, L=2, prefill=14, query_width=4, logits="normal"),
    scaled(C4, T=20, k=4, E=16, H=64, I=64, S=30, L=2, prefill=20, query_width=8),
], ids=["c1", "bf16_small", "nvfp4_small"])
def test_slot_path_equals_stream_path(cfg):
    src, cache, pool = _slot_setup(cfg)
    a = forward_slots(cfg, router_inputs(cfg), lambda l, e: src[l][e], cache, pool, block=4)
    b = forward_stream(cfg, router_inputs(cfg), lambda e: src[cfg.layer][e], block=4)
    assert a["ok"]
    assert np.array_equal(a["out"], b["out"])
    assert np.array_equal(a["sorted_ids"], b["sorted_ids"])
    for e in range(cfg.E):
        if e in set(a["ids"].reshape(-1).tolist()):
            assert a["e2s"][e] >= 0


def test_160_experts_take_queries_of_128_and_32():
    cfg = scaled(C1, T=96, k=2, E=160, H=64, I=64, S=200, L=1, prefill=0, query_width=128,
                 logits="normal")
    rin = router_inputs(cfg)
    # route token t to experts (2t, 2t+1) mod 160: 160 distinct experts
    logits = np.full((cfg.T, cfg.E), -10.0, dtype=np.float32)
    for t in range(cfg.T):
        logits[t, (2 * t) % 160] = 1.0
        logits[t, (2 * t + 1) % 160] = 0.5
    rin["logits"] = logits
    src, cache, pool = _slot_setup(cfg)
    res = forward_slots(cfg, rin, lambda l, e: src[l][e], cache, pool, block=16)
    assert res["D"] == 160
    assert [len([k for k in q["keys"] if k >= 0]) for q in res["queries"]] == [128, 32]
    assert [len(q["misses"]) for q in res["queries"]] == [128, 32]
    for q in res["queries"]:
        for key, slot, _ in q["misses"]:
            assert np.array_equal(pool[slot], src[0][key])
    assert cache.stats() == {"hits": 0, "misses": 0, "evictions": 0}
    assert not cache.decode_freq.any()


def test_resident_rows_untouched():
    cfg = scaled(C1, T=24, k=3, E=12, H=64, I=64, S=20, L=2, prefill=14, query_width=4,
                 logits="normal")
    src, cache, pool = _slot_setup(cfg)
    before = dict(pool)
    res = forward_slots(cfg, router_inputs(cfg), lambda l, e: src[l][e], cache, pool, block=4)
    written = {slot for q in res["queries"] for _, slot, _ in q["misses"]}
    for s in range(cfg.S):
        if s not in written:
            assert pool[s] is before[s]
