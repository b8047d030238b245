"""GPU parity of the whole layer: the grouped GEMM over the slot pool and the
streamed path, against the oracle.

* Bit-exact: routed ids, distinct list, align outputs, slot-cache tables.
* Layer output vs the oracle (fp64): max-abs <= 2e-2 and rel-L2 <= 5e-3 for
  bf16 weights, <= 5e-2 and <= 1e-2 for NVFP4 weights.  The GPU rounds h
  (16-bit), y (bf16) and out (bf16); the oracle keeps fp64 throughout.
* Slot path == streamed path, byte for byte (FreeToken PR #676, Solution).
* A demand admission records no statistic; a chunk the pool cannot hold is
  refused and streams.
"""
import numpy as np
import pytest
import torch

from gpu_util import Workload, bf16_to_f64, lib, rel_l2, scratch, status
from offloaded_expert_slot_gb300 import oes
from offloaded_expert_slot_gb300.configs import C1, C2, C3, C4, C5, scaled
from oracle.layer import forward_slots, forward_stream
from oracle.slot_cache import SlotCache

pytestmark = pytest.mark.gpu

TOL = {"bf16": (2e-2, 5e-3), "nvfp4": (5e-2, 1e-2)}

MEDIUM_BF16 = scaled(C2, name="medium_bf16", T=96, k=4, E=16, H=256, I=192, S=40, L=2, prefill=20,
                     query_width=128)
MEDIUM_NVFP4 = scaled(C4, name="medium_nvfp4", T=96, k=4, E=16, H=256, I=192, S=40, L=2, prefill=20)
WIDE_BLOCKS = scaled(C2, name="wide_blocks_bf16", T=160, k=8, E=12, H=128, I=128, S=30, L=2,
                     prefill=10)
# NVFP4 blocks of more than 96 routes (a unit then takes both of the NVFP4
# kernel's accumulator slots), a GEMM2 tile pair whose second tile lies past
# H, and K loops of two chunks
WIDE_BLOCKS_NVFP4 = scaled(C4, name="wide_blocks_nvfp4", T=160, k=8, E=12, H=128, I=128, S=30,
                           L=2, prefill=10)
# few routes per expert: blocks of 16 on the weight-major kernel, ragged I
MEDIUM_SWAP_BF16 = scaled(C2, name="medium_swap_bf16", T=40, k=3, E=16, H=256, I=192, S=40, L=2,
                          prefill=20)
MEDIUM_SWAP_NVFP4 = scaled(C4, name="medium_swap_nvfp4", T=40, k=3, E=16, H=256, I=192, S=40,
                           L=2, prefill=20)


def desc_of(cfg):
    return oes.layer_desc(cfg.E, cfg.H, cfg.I, oes.OES_WFMT_BF16 if cfg.wfmt == "bf16"
                          else oes.OES_WFMT_NVFP4)


GUARD_ROWS = 2
GUARD_BITS = 0x7FA5                 # a bf16 NaN pattern no kernel writes


class Run:
    def __init__(self, w: Workload):
        cfg = w.cfg
        self.desc = desc_of(cfg)
        self.wsb = oes.moe_layer_workspace_size(self.desc, cfg.T, cfg.k)
        self.ws = scratch(self.wsb)
        # the output between canary rows that no call may touch
        self.out_all = torch.full((cfg.T + 2 * GUARD_ROWS, cfg.H), GUARD_BITS, dtype=torch.int16,
                                  device="cuda").view(torch.bfloat16)
        self.out = self.out_all[GUARD_ROWS:GUARD_ROWS + cfg.T]
        self.out.zero_()
        self.status = status()
        self.chunk = oes.chunk(w.x, cfg.T, cfg.k, self.out, self.status, self.ws, self.wsb,
                               logits=w.logits, gate=w.gate)

    def guards_intact(self) -> bool:
        g = torch.cat([self.out_all[:GUARD_ROWS], self.out_all[GUARD_ROWS + self.out.shape[0]:]])
        return bool((g.view(torch.int16) == GUARD_BITS).all())

    def views(self, cfg):
        v = oes.moe_layer_workspace_views(self.desc, cfg.T, cfg.k, self.ws)
        R = cfg.T * cfg.k
        B = oes.oes_tile_plan(R, cfg.E)
        cap = oes.align_capacity(R, cfg.E, B)

        def arr(ptr, n, dtype):
            base = self.ws.data_ptr()
            off = ptr - base
            nbytes = n * np.dtype(dtype).itemsize
            return self.ws[off:off + nbytes].cpu().numpy().view(dtype)

        return {"ids": arr(v["ids"], R, np.int32).reshape(cfg.T, cfg.k),
                "weights": arr(v["weights"], R, np.float32).reshape(cfg.T, cfg.k),
                "distinct": arr(v["distinct"], min(R, cfg.E), np.int32),
                "sorted_ids": arr(v["sorted_ids"], cap, np.int32),
                "block_expert": arr(v["block_expert"], cap // B, np.int32),
                "n_post_pad": int(arr(v["n_post_pad"], 1, np.int32)[0])}


def gpu_slots(w: Workload, layer=None, record_stats=False):
    r = Run(w)
    layer = w.cfg.layer if layer is None else layer
    oes.moe_layer_forward_slots(w.cache, w.src, w.pool, layer, r.desc, r.chunk, record_stats)
    torch.cuda.synchronize()
    assert r.guards_intact(), "output canary rows were written"
    return r


def gpu_stream(w: Workload, layer=None, two_streams=True):
    cfg = w.cfg
    r = Run(w)
    layer = cfg.layer if layer is None else layer
    buf = torch.empty((cfg.E, cfg.row_bytes), dtype=torch.uint8, device="cuda")
    cs = torch.cuda.Stream() if two_streams else None
    oes.moe_layer_forward_stream(w.src, buf, layer, r.desc, r.chunk, copy_stream=cs)
    torch.cuda.synchronize()
    assert r.guards_intact(), "output canary rows were written"
    return r


def oracle_slots(w: Workload, tokens=None, layer=None):
    cfg = w.cfg
    st = w.prefill
    cache = SlotCache.from_state(cfg.S, cfg.L, cfg.E, st["slot_key"], st["slot_ts"], st["clock"])
    B = oes.oes_tile_plan(cfg.T * cfg.k, cfg.E)
    res = forward_slots(cfg, w.rin, w.source_row, cache, w.oracle_pool(), block=B, layer=layer,
                        tokens=tokens)
    return res, cache


def check_close(got: torch.Tensor, want: np.ndarray, wfmt: str, rows=None):
    g = bf16_to_f64(got)
    if rows is not None:
        g, want = g[rows], want[rows]
    amax, rl2 = TOL[wfmt]
    err = np.abs(g - want).max()
    rl = rel_l2(g, want)
    assert np.isfinite(g).all()
    assert err <= amax and rl <= rl2, (err, rl)
    return err, rl


def full_check(w: Workload, tokens=None):
    cfg = w.cfg
    r = gpu_slots(w)
    assert int(r.status.item()) == 0
    o, ocache = oracle_slots(w, tokens=tokens)
    v = r.views(cfg)
    assert np.array_equal(v["ids"], o["ids"])
    np.testing.assert_allclose(v["weights"], o["w"], rtol=2e-6, atol=1e-7)
    assert np.array_equal(v["distinct"], o["distinct"])
    assert v["n_post_pad"] == o["n_post_pad"]
    assert np.array_equal(v["sorted_ids"], o["sorted_ids"])
    assert np.array_equal(v["block_expert"], o["block_expert"])
    st = oes.slot_cache_read_state(w.cache, cfg.S, cfg.L, cfg.E)
    assert np.array_equal(st["map"], ocache.map)
    assert np.array_equal(st["slot_key"], ocache.slot_key)
    assert np.array_equal(st["slot_ts"], ocache.slot_ts)
    assert st["hits"] == st["misses"] == st["evictions"] == 0 and not st["decode_freq"].any()
    rows = None if tokens is None else np.asarray(tokens)
    check_close(r.out, o["out"], cfg.wfmt, rows)
    s = gpu_stream(w)
    assert int(s.status.item()) == 0
    assert torch.equal(s.out.view(torch.int16), r.out.view(torch.int16)), "slot != stream"
    return r


@pytest.mark.parametrize("cfg", [MEDIUM_BF16, WIDE_BLOCKS, MEDIUM_NVFP4, WIDE_BLOCKS_NVFP4,
                                 MEDIUM_SWAP_BF16, MEDIUM_SWAP_NVFP4], ids=lambda c: c.name)
def test_medium_layers_match_oracle_and_stream(cfg):
    """Several tiles with a ragged last tile (I = 192), several K chunks,
    experts with several blocks and ragged block tails, on both kernels
    (token-major for many routes per expert, weight-major for few)."""
    lib()
    R = cfg.T * cfg.k
    assert oes.oes_tile_plan(R, cfg.E) == (16 if "swap" in cfg.name else 128)
    w = Workload(cfg, gen_device="cpu")
    full_check(w)
    w.close()


@pytest.mark.parametrize("prefill", [47, 46, 45, 30, 0])
def test_two_part_copies(prefill):
    """One query of 48 ids, more than the 32 above which a query's misses are
    copied in two launches (the last min(n/2, 16) second), each with its own
    GEMM: 1, 2, 3, 18 and 48 misses put the split at its edges (an empty
    second part, a one-miss part, a full 16-miss part)."""
    lib()
    cfg = scaled(C2, name=f"split_bf16_p{prefill}", T=40, k=6, E=48, H=128, I=128, S=60, L=1,
                 prefill=prefill)
    w = Workload(cfg, gen_device="cpu")
    o, _ = oracle_slots(w)
    assert len(o["distinct"]) == 48 and (np.asarray(o["distinct"]) >= 0).all()
    r = full_check(w)
    st = oes.slot_cache_read_state(w.cache, cfg.S, cfg.L, cfg.E)
    assert int((st["slot_key"] >= 0).sum()) == 48           # prefill + misses, all of layer 0
    w.close()


def test_full_pool_two_queries():
    """Every slot full and two queries: query 1's misses evict the oldest
    slots, some holding experts of query 2 that were resident before the
    chunk; the overlapped GEMM must only take experts that were hits in their
    own query (tables, output and slot == stream as everywhere)."""
    lib()
    cfg = scaled(C2, name="full_pool_bf16", T=40, k=4, E=512, H=256, I=192, S=200, L=2,
                 prefill=200)
    w = Workload(cfg, gen_device="cpu")
    o, _ = oracle_slots(w)
    q1 = {k_ for k_, _s, _old in o["queries"][0]["misses"]}
    evicted = {old for q in o["queries"][:1] for _k, _s, old in q["misses"] if old >= 0}
    later = {int(k_) for q in o["queries"][1:] for k_ in q["keys"] if k_ >= 0}
    assert len(o["queries"]) >= 2 and q1 and evicted & later, "the case must evict a later query's expert"
    full_check(w)
    w.close()


def test_tiny_workload_streams_and_is_refused_by_slots():
    lib()
    w = Workload(C1, gen_device="cpu")
    r = Run(w)
    with pytest.raises(oes.OesError) as e:
        oes.moe_layer_forward_slots(w.cache, w.src, w.pool, 0, r.desc, r.chunk, 0)
    assert e.value.code == oes.OES_ERR_CAPACITY
    s = gpu_stream(w)
    assert int(s.status.item()) == 0
    o = forward_stream(C1, w.rin, lambda e: w.source_row(0, e), block=16)
    check_close(s.out, o["out"], "bf16")
    w.close()


def test_slot_path_over_small_pool_equals_large_pool():
    """The same chunk over a pool of exactly the layer's experts and over a
    pool with many foreign slots gives the same bytes (tiles sized by the
    layer's experts, not the slots)."""
    lib()
    a = Workload(scaled(MEDIUM_BF16, S=16, L=1, prefill=0), gen_device="cpu")
    b = Workload(scaled(MEDIUM_BF16, S=200, L=1, prefill=0), gen_device="cpu")
    ra, rb = gpu_slots(a), gpu_slots(b)
    assert torch.equal(ra.out.view(torch.int16), rb.out.view(torch.int16))
    a.close()
    b.close()


def test_record_stats_counts_decode_admissions():
    lib()
    w = Workload(MEDIUM_BF16, gen_device="cpu")
    gpu_slots(w, record_stats=True)
    o, oc = oracle_slots(w)
    cfg = w.cfg
    oc2 = SlotCache.from_state(cfg.S, cfg.L, cfg.E, w.prefill["slot_key"], w.prefill["slot_ts"],
                               w.prefill["clock"])
    for q in o["queries"]:
        oc2.ensure(q["keys"], record_stats=True)
    st = oes.slot_cache_read_state(w.cache, cfg.S, cfg.L, cfg.E)
    assert (st["hits"], st["misses"], st["evictions"]) == (oc2.hits, oc2.misses, oc2.evictions)
    assert np.array_equal(st["decode_freq"], oc2.decode_freq)
    assert st["misses"] > 0
    w.close()


@pytest.mark.parametrize("cfg,tokens", [(C2, None), (C3, None), (C4, 40)],
                         ids=["c2_decode_width", "c3_short_prefill", "c4_nvfp4_prefill"])
def test_workload_layers(cfg, tokens):
    lib()
    w = Workload(cfg)
    toks = None if tokens is None else np.random.default_rng(4).choice(cfg.T, tokens, replace=False)
    full_check(w, tokens=toks)
    if cfg.wfmt == "nvfp4":
        # the view must carry the layer's input scales, not a slot's (FreeToken
        # PR #676, Tests: 9.0 in every other slot against the layer's 2.0 / 3.0)
        from oracle.expert_mlp import input_scales
        layer_scale = cfg.layer_input_scales[cfg.layer]
        for e in (0, 7, 511):
            assert input_scales(w.source_row(cfg.layer, e), cfg.H, cfg.I) == (layer_scale, layer_scale)
        empties = np.nonzero(w.prefill["slot_key"] < 0)[0]
        row = w.pool[int(empties[-1])].cpu().numpy()
        st = oes.slot_cache_read_state(w.cache, cfg.S, cfg.L, cfg.E)
        if st["slot_key"][int(empties[-1])] < 0:
            assert input_scales(row, cfg.H, cfg.I) == (9.0, 9.0)
    w.close()


@pytest.mark.parametrize("cfg", [scaled(C2, name="one_token_bf16", T=1),
                                 scaled(C4, name="one_token_nvfp4", T=1),
                                 scaled(C2, name="two_tokens_bf16", T=2)], ids=lambda c: c.name)
def test_few_token_decode(cfg):
    """One token x top-10 over the decode-width layer (512 experts, hidden
    2048, intermediate 768): GEMM1's 60 tiles fill at most half the SMs, so
    each tile's K range is shared by two CTAs and the second to finish writes
    h.  Two tokens (120 tiles) take whole tiles.  Either way slot == stream
    byte for byte and the output follows the oracle; a second, warm call (every
    expert a hit, the GEMM over the hits alone) gives the same bytes."""
    lib()
    w = Workload(cfg)
    first = full_check(w)
    warm = gpu_slots(w)
    assert int(warm.status.item()) == 0
    assert torch.equal(warm.out.view(torch.int16), first.out.view(torch.int16))
    w.close()


def _one_token_out(w: Workload, layer: int, ids: np.ndarray, wts: np.ndarray, t: int) -> np.ndarray:
    """The oracle's output row of token t of a layer: its k experts' SwiGLU
    MLPs on the layer's source rows (the rows its slots hold), combined in
    j order, in fp64."""
    from oracle.expert_mlp import expert_weights, swiglu_expert
    from oracle.numerics import bf16_to_f64 as obf16
    cfg = w.cfg
    x = obf16(w.rin["x"][t])[None]
    acc = np.zeros(cfg.H)
    for j in range(cfg.k):
        w13, w2 = expert_weights(w.source_row(layer, int(ids[t, j])), cfg.wfmt, cfg.H, cfg.I)
        acc += np.float64(wts[t, j]) * swiglu_expert(x, w13, w2)[0]
    return acc


def test_long_prefill_layers_sequence():
    """4096 tokens x top-10 over 48 layers of 512 NVFP4 experts in a
    1650-slot pool: all 48 layers forwarded in turn through the slot path
    (each evicting older layers' experts) and the streamed path, slot ==
    stream byte for byte on every layer.  On every layer the tables follow
    the oracle's LRU bit for bit and one token's output row (a different
    token per layer) follows the oracle's MLP; layers 0 and 2 also run the
    oracle's whole slot path on 12 sampled tokens."""
    from oracle.distinct import distinct_experts
    from oracle.layer import route
    lib()
    cfg = C5
    w = Workload(cfg)
    R = cfg.T * cfg.k
    assert oes.oes_tile_plan(R, cfg.E) == 128
    toks = np.random.default_rng(5).choice(cfg.T, 12, replace=False)
    one = np.random.default_rng(6).choice(cfg.T, cfg.L, replace=False)
    ocache = SlotCache.from_state(cfg.S, cfg.L, cfg.E, w.prefill["slot_key"], w.prefill["slot_ts"],
                                  w.prefill["clock"])
    opool = w.oracle_pool()
    _l, oids, ow = route(w.rin, cfg.k)
    odist, _D = distinct_experts(oids, cfg.E)
    for layer in range(cfg.L):
        r = gpu_slots(w, layer=layer)
        assert int(r.status.item()) == 0, layer
        s = gpu_stream(w, layer=layer)
        assert torch.equal(s.out.view(torch.int16), r.out.view(torch.int16)), layer
        if layer in (0, 2):
            o = forward_slots(cfg, w.rin, w.source_row, ocache, opool, block=128, layer=layer,
                              tokens=toks)
            assert o["ok"]
            check_close(r.out, o["out"], "nvfp4", toks)
        else:
            for q0 in range(0, odist.size, cfg.query_width):
                keys = [layer * cfg.E + int(e) if e >= 0 else -1
                        for e in odist[q0:q0 + cfg.query_width]]
                assert ocache.ensure(keys)[0] == 0
        st = oes.slot_cache_read_state(w.cache, cfg.S, cfg.L, cfg.E)
        assert np.array_equal(st["map"], ocache.map), layer
        assert np.array_equal(st["slot_key"], ocache.slot_key), layer
        assert np.array_equal(st["slot_ts"], ocache.slot_ts), layer
        t = int(one[layer])
        want = _one_token_out(w, layer, oids, ow, t)
        check_close(r.out[t:t + 1], want[None], "nvfp4")
    w.close()


def test_demand_token_dispatch():
    """FreeToken PR #676, Solution and Tests: with threshold N a chunk of at
    most N tokens goes through the slot cache, a longer one (or any chunk at
    N = 0) streams and leaves the cache alone; both give the same bytes; a
    chunk the pool cannot hold streams at any threshold."""
    lib()
    cfg = MEDIUM_SWAP_BF16
    w = Workload(cfg, gen_device="cpu")
    st0 = oes.slot_cache_read_state(w.cache, cfg.S, cfg.L, cfg.E)
    outs = {}
    for N, want_slots in [(0, False), (cfg.T - 1, False), (cfg.T, True)]:
        r = Run(w)
        buf = torch.empty((cfg.E, cfg.row_bytes), dtype=torch.uint8, device="cuda")
        took = oes.moe_layer_forward(w.cache, w.src, w.pool, buf, cfg.layer, r.desc, r.chunk, N, 0,
                                     copy_stream=torch.cuda.Stream())
        torch.cuda.synchronize()
        assert took == want_slots and int(r.status.item()) == 0
        st = oes.slot_cache_read_state(w.cache, cfg.S, cfg.L, cfg.E)
        if not want_slots:
            assert np.array_equal(st["slot_key"], st0["slot_key"])
            assert np.array_equal(st["slot_ts"], st0["slot_ts"])
        outs[N] = r.out.view(torch.int16).clone()
    o, ocache = oracle_slots(w)
    st = oes.slot_cache_read_state(w.cache, cfg.S, cfg.L, cfg.E)
    assert np.array_equal(st["slot_key"], ocache.slot_key)
    assert np.array_equal(st["map"], ocache.map)
    assert torch.equal(outs[0], outs[cfg.T]) and torch.equal(outs[0], outs[cfg.T - 1])
    check_close(outs[cfg.T].view(torch.bfloat16), o["out"], "bf16")
    w.close()

    t = Workload(C1, gen_device="cpu")
    r = Run(t)
    buf = torch.empty((C1.E, C1.row_bytes), dtype=torch.uint8, device="cuda")
    assert not oes.moe_layer_forward(t.cache, t.src, t.pool, buf, 0, r.desc, r.chunk, 1 << 20, 0)
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0
    t.close()
