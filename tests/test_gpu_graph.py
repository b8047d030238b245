"""The decode step as one CUDA graph (route -> distinct -> ensures with
decode statistics -> miss copies -> grouped GEMM -> combine), captured once
and replayed on new tokens with no host code in between.

Three decode steps of different tokens are replayed from one capture on one
cache; the same steps run eagerly on a second cache with the same pre-fill,
and through the oracle.  Checked: output bytes graph == eager; tables,
counters and decode_freq graph == eager == oracle, bit for bit; output vs the
oracle within the bf16 layer tolerance; every step leaves status 0.
"""
import numpy as np
import pytest
import torch

from gpu_util import Workload, bits16, cuda, lib
from offloaded_expert_slot_gb300 import oes
from offloaded_expert_slot_gb300.configs import C2, scaled
from offloaded_expert_slot_gb300.inputs import router_inputs
from oracle.layer import forward_slots
from oracle.slot_cache import SlotCache
from test_gpu_layer import Run, check_close

pytestmark = pytest.mark.gpu

# two queries per step (about 200 distinct experts of 300), 320 slots over two layers
GRAPH_DECODE = scaled(C2, name="graph_decode", T=40, k=8, E=300, H=256, I=192, S=320, L=2,
                      prefill=200)
STEPS = 3


def step_inputs(cfg, s):
    return router_inputs(scaled(cfg, seed=cfg.seed + 101 * s))


def load_step(w, rin):
    w.x.copy_(bits16(rin["x"]))
    w.logits.copy_(cuda(rin["logits"]))


def tables(w):
    cfg = w.cfg
    return oes.slot_cache_read_state(w.cache, cfg.S, cfg.L, cfg.E)


@pytest.mark.parametrize("policy", ["lru", "lrfu"])
def test_decode_step_graph_replays_match_eager_and_oracle(policy):
    """Under LRFU each replay must draw a fresh chunk pin tag on the device,
    as each eager call does; a tag fixed in the graph would leave the last
    step's pins in force."""
    lib()
    cfg = GRAPH_DECODE
    k = 3

    def set_policy(w):
        if policy == "lrfu":
            oes.slot_cache_set_policy(w.cache, oes.OES_POLICY_LRFU, k)
    ins = [step_inputs(cfg, s) for s in range(STEPS)]

    # eager reference on its own cache
    we = Workload(cfg, gen_device="cpu")
    set_policy(we)
    re_ = Run(we)
    eager_out, eager_tab = [], []
    for rin in ins:
        load_step(we, rin)
        oes.moe_layer_forward_slots(we.cache, we.src, we.pool, cfg.layer, re_.desc, re_.chunk, 1)
        torch.cuda.synchronize()
        assert int(re_.status.item()) == 0
        eager_out.append(re_.out.clone())
        eager_tab.append(tables(we) | dict(zip(("crf", "pin"), oes.slot_cache_read_lrfu(we.cache,
                                                                                      cfg.S))))

    # graph: one eager warm-up (one-time kernel attributes), back to the pre-fill, capture
    wg = Workload(cfg, gen_device="cpu")
    set_policy(wg)
    rg = Run(wg)
    load_step(wg, ins[0])
    oes.moe_layer_forward_slots(wg.cache, wg.src, wg.pool, cfg.layer, rg.desc, rg.chunk, 1)
    torch.cuda.synchronize()
    wg.reset_pool()
    rg.status.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        oes.moe_layer_forward_slots(wg.cache, wg.src, wg.pool, cfg.layer, rg.desc, rg.chunk, 1)
    torch.cuda.synchronize()
    assert tables(wg)["clock"] == wg.prefill["clock"], "capture must not run the step"

    ocache = SlotCache.from_state(cfg.S, cfg.L, cfg.E, wg.prefill["slot_key"],
                                  wg.prefill["slot_ts"], wg.prefill["clock"])
    if policy == "lrfu":
        ocache.set_policy("lrfu", k)
    opool = wg.oracle_pool()
    B = oes.oes_tile_plan(cfg.T * cfg.k, cfg.E)
    n_queries = []
    for s, rin in enumerate(ins):
        load_step(wg, rin)
        g.replay()
        torch.cuda.synchronize()
        assert int(rg.status.item()) == 0
        assert torch.equal(rg.out.view(torch.int16), eager_out[s].view(torch.int16)), s
        t = tables(wg)
        t |= dict(zip(("crf", "pin"), oes.slot_cache_read_lrfu(wg.cache, cfg.S)))
        for key in ("map", "slot_key", "slot_ts", "decode_freq", "crf", "pin"):
            assert np.array_equal(t[key], eager_tab[s][key]), (s, key)
        o = forward_slots(scaled(cfg, seed=cfg.seed + 101 * s), rin, wg.source_row, ocache, opool,
                          block=B, record_stats=True, tag=s + 1)
        n_queries.append(len(o["queries"]))
        assert np.array_equal(t["map"], ocache.map) and np.array_equal(t["slot_ts"], ocache.slot_ts)
        assert np.array_equal(t["decode_freq"], ocache.decode_freq)
        assert [int(v) for v in t["crf"]] == ocache.crf and [int(v) for v in t["pin"]] == ocache.pin
        assert (t["hits"], t["misses"], t["evictions"]) == (ocache.hits, ocache.misses,
                                                          ocache.evictions)
        check_close(rg.out, o["out"], "bf16")
    assert min(n_queries) >= 2 and ocache.misses > 0 and ocache.evictions > 0
    del g
    we.close()
    wg.close()
