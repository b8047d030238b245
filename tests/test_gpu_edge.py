"""Degenerate and maximum-size cases of the layer path, through the C ABI.

* An empty chunk (T = 0) on every composite: OK, nothing written, the cache
  unchanged.
* One token, one route, one expert (T = k = E = 1).
* k = E: every token routes to every expert.
* The same chunk twice: the second call has no miss in any query, gives the
  same bytes, and the tables follow the oracle through both calls.
* The largest layer: E = 4096 experts at top-32, 2048 tokens, so all 4096
  experts are routed, in 32 queries of 128, over a pool of exactly 4096
  slots.
"""
import numpy as np
import pytest
import torch

from gpu_util import Workload, lib, scratch, status
from offloaded_expert_slot_gb300 import oes
from offloaded_expert_slot_gb300.configs import C2, scaled
from oracle.layer import forward_slots
from oracle.slot_cache import SlotCache
from test_gpu_layer import Run, check_close, gpu_stream, oracle_slots

pytestmark = pytest.mark.gpu


def small(name, **kw):
    base = dict(T=24, k=4, E=16, H=128, I=64, S=40, L=2, prefill=10)
    base.update(kw)
    return scaled(C2, name=name, **base)


def tables(w):
    cfg = w.cfg
    return oes.slot_cache_read_state(w.cache, cfg.S, cfg.L, cfg.E)


def test_empty_chunk_everywhere():
    lib()
    cfg = small("empty", T=0)
    w = Workload(cfg, gen_device="cpu", extra_rows=2 * cfg.E)
    before = tables(w)
    desc = oes.layer_desc(cfg.E, cfg.H, cfg.I, oes.OES_WFMT_BF16)
    wsb = max(oes.moe_layer_workspace_size(desc, 0, cfg.k), 256)
    ws = scratch(wsb)
    out = torch.full((1, cfg.H), 7.0, dtype=torch.bfloat16, device="cuda")
    st = status()
    x = torch.zeros((1, cfg.H), dtype=torch.int16, device="cuda")
    lg = torch.zeros((1, cfg.E), dtype=torch.float32, device="cuda")
    ch = oes.chunk(x, 0, cfg.k, out, st, ws, wsb, logits=lg)
    buf = torch.empty((cfg.E, cfg.row_bytes), dtype=torch.uint8, device="cuda")
    oes.moe_layer_forward_slots(w.cache, w.src, w.pool, 0, desc, ch, 1)
    oes.moe_layer_forward_stream(w.src, buf, 0, desc, ch)
    assert not oes.moe_layer_forward(w.cache, w.src, w.pool, buf, 0, desc, ch, 512, 1)
    plan = oes.oes_stage_plan_create(w.cache, [0, 1], True)
    oes.moe_layers_forward_staged(plan, w.src, w.pool_all, desc, [ch, ch])
    torch.cuda.synchronize()
    oes.oes_stage_plan_destroy(plan)
    assert int(st.item()) == 0
    assert (out.float() == 7.0).all()
    after = tables(w)
    for key in ("map", "slot_key", "slot_ts", "clock", "hits", "misses", "decode_freq"):
        assert np.array_equal(np.asarray(after[key]), np.asarray(before[key])), key
    w.close()


@pytest.mark.parametrize("cfg", [small("one_route", T=1, k=1, E=1, S=4, L=1, prefill=0),
                                 small("k_equals_E", T=16, k=8, E=8, S=20, L=2, prefill=6)],
                         ids=lambda c: c.name)
def test_degenerate_routings(cfg):
    lib()
    w = Workload(cfg, gen_device="cpu")
    r = Run(w)
    oes.moe_layer_forward_slots(w.cache, w.src, w.pool, cfg.layer, r.desc, r.chunk, 0)
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    o, oc = oracle_slots(w)
    if cfg.k == cfg.E:
        assert (np.sort(o["ids"], axis=1) == np.arange(cfg.E)).all()
    t = tables(w)
    assert np.array_equal(t["map"], oc.map) and np.array_equal(t["slot_ts"], oc.slot_ts)
    check_close(r.out, o["out"], "bf16")
    s = gpu_stream(w)
    assert torch.equal(s.out.view(torch.int16), r.out.view(torch.int16))
    w.close()


def test_second_call_has_no_misses():
    lib()
    cfg = small("twice", T=48, k=6, E=64, S=100, L=2, prefill=30)
    w = Workload(cfg, gen_device="cpu")
    r = Run(w)
    outs = []
    for _ in range(2):
        oes.moe_layer_forward_slots(w.cache, w.src, w.pool, cfg.layer, r.desc, r.chunk, 1)
        torch.cuda.synchronize()
        assert int(r.status.item()) == 0
        outs.append(r.out.clone())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    st0 = w.prefill
    oc = SlotCache.from_state(cfg.S, cfg.L, cfg.E, st0["slot_key"], st0["slot_ts"], st0["clock"])
    pool = w.oracle_pool()
    B = oes.oes_tile_plan(cfg.T * cfg.k, cfg.E)
    forward_slots(cfg, w.rin, w.source_row, oc, pool, block=B, record_stats=True)
    misses_first = oc.misses
    o2 = forward_slots(cfg, w.rin, w.source_row, oc, pool, block=B, record_stats=True)
    assert misses_first > 0 and oc.misses == misses_first          # none the second time
    assert all(not q["misses"] for q in o2["queries"])
    t = tables(w)
    assert (t["hits"], t["misses"], t["evictions"]) == (oc.hits, oc.misses, oc.evictions)
    assert np.array_equal(t["slot_ts"], oc.slot_ts) and np.array_equal(t["decode_freq"], oc.decode_freq)
    check_close(outs[1], o2["out"], "bf16")
    w.close()


def test_largest_layer_32_queries():
    """E = 4096 (the largest), top-32 (the largest), 2048 tokens: all 4096
    experts routed, 32 queries, pool of exactly 4096 slots; tables bit-exact,
    sampled tokens against the oracle, slot == stream."""
    lib()
    cfg = scaled(C2, name="largest", T=2048, k=32, E=4096, H=64, I=64, S=4096, L=1, prefill=0)
    w = Workload(cfg, gen_device="cpu")
    r = Run(w)
    oes.moe_layer_forward_slots(w.cache, w.src, w.pool, 0, r.desc, r.chunk, 0)
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    toks = np.random.default_rng(9).choice(cfg.T, 16, replace=False)
    o, oc = oracle_slots(w, tokens=toks)
    assert o["D"] == 4096 and len(o["queries"]) == 32
    t = tables(w)
    assert np.array_equal(t["map"], oc.map) and np.array_equal(t["slot_key"], oc.slot_key)
    check_close(r.out, o["out"], "bf16", rows=toks)
    s = gpu_stream(w)
    assert torch.equal(s.out.view(torch.int16), r.out.view(torch.int16))
    w.close()


def test_two_host_threads_two_caches():
    """The library is re-entrant across caches: two host threads, each with
    its own cache, pool and stream, run the slot path at the same time
    (ctypes releases the interpreter lock) and each gets exactly the bytes a
    lone run gives."""
    import threading
    lib()
    cfgs = [small("thread_a", T=32, k=4, E=64, S=80, L=2, prefill=30, seed=2101),
            small("thread_b", T=48, k=6, E=64, S=80, L=2, prefill=50, seed=2102)]
    want = []
    for cfg in cfgs:
        w = Workload(cfg, gen_device="cpu")
        r = Run(w)
        oes.moe_layer_forward_slots(w.cache, w.src, w.pool, 0, r.desc, r.chunk, 1)
        torch.cuda.synchronize()
        want.append(r.out.view(torch.int16).clone())
        w.close()
    works = [Workload(cfg, gen_device="cpu") for cfg in cfgs]
    runs = [Run(w) for w in works]
    errors = []

    def worker(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                oes.moe_layer_forward_slots(works[i].cache, works[i].src, works[i].pool, 0,
                                            runs[i].desc, runs[i].chunk, 1)
            s.synchronize()
        except Exception as e:            # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for i in range(2):
        assert int(runs[i].status.item()) == 0
        assert torch.equal(runs[i].out.view(torch.int16), want[i]), i
        works[i].close()


@pytest.mark.parametrize("wfmt,T", [("bf16", 8), ("bf16", 24), ("nvfp4", 8)],
                         ids=["bf16_weight_major", "bf16_token_major", "nvfp4_weight_major"])
def test_wide_layer(wfmt, T):
    """H = 8192, I = 4096: 128 K chunks per GEMM1 tile and 64 (weight-major)
    or 32 (token-major) output tiles in GEMM2, on 4 experts; every token
    against the oracle, slot == stream.  The outputs here are about 3x the
    workloads' (sums over 8192 and 4096 terms), so the max-abs bar scales
    with them: the GPU rounds h, y and out to 16 bits (each within 2^-9 of
    the value, NVFP4's h f16 and bf16 y), and h's rounding adds noise over
    the 4096-term down projection, so max-abs <= 2^-7 * max|out| (rel-L2
    keeps the layer bar)."""
    from offloaded_expert_slot_gb300.configs import C4
    lib()
    base = C2 if wfmt == "bf16" else C4
    cfg = scaled(base, name=f"wide_{wfmt}_{T}", T=T, k=2, E=4, H=8192, I=4096, S=6, L=1,
                 prefill=0)
    w = Workload(cfg, gen_device="cpu")
    r = Run(w)
    oes.moe_layer_forward_slots(w.cache, w.src, w.pool, 0, r.desc, r.chunk, 0)
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    assert oes.oes_tile_plan(T * 2, 4) == (128 if T == 24 else 16)
    o, _oc = oracle_slots(w)
    got = r.out.to(torch.float64).cpu().numpy()
    want = o["out"]
    err = float(np.abs(got - want).max())
    rl2 = float(np.linalg.norm(got - want) / np.linalg.norm(want))
    bar = 5e-3 if wfmt == "bf16" else 1e-2
    assert np.isfinite(got).all()
    assert err <= 2.0 ** -7 * np.abs(want).max() and rl2 <= bar, (err, np.abs(want).max(), rl2)
    s = gpu_stream(w)
    assert torch.equal(s.out.view(torch.int16), r.out.view(torch.int16))
    w.close()
