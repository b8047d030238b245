"""GPU parity of prefill staging over a layer sequence (vLLM fork PR #51,
Details, and its staging test), through the C ABI.

* The plan's runs and staged-row counts equal the oracle's, bit for bit,
  on the cache's real placement.
* Every layer's output equals moe_layer_forward_stream's for that layer,
  byte for byte, and the oracle's within the layer tolerance.
* The cache's slots are untouched; the last staging buffer holds the
  source rows of exactly the experts staged into it.
* Four layers through two buffers, so each buffer is reused after the
  compute that read it.
"""
import numpy as np
import pytest
import torch

from gpu_util import Workload, lib
from offloaded_expert_slot_gb300 import oes
from offloaded_expert_slot_gb300.configs import C2, C4, scaled
from oracle.slot_cache import SlotCache
from oracle.stage import forward_staged_layers, stage_runs, staged_pool
from test_gpu_layer import Run, check_close, gpu_stream

pytestmark = pytest.mark.gpu

STAGE_BF16 = scaled(C2, name="stage_bf16", T=96, k=4, E=16, H=256, I=192, S=24, L=3, prefill=14)
STAGE_NVFP4 = scaled(C4, name="stage_nvfp4", T=40, k=3, E=16, H=256, I=192, S=24, L=3, prefill=14)


@pytest.mark.parametrize("skip", [True, False], ids=["skip_resident", "whole_layer"])
@pytest.mark.parametrize("cfg", [STAGE_BF16, STAGE_NVFP4], ids=lambda c: c.name)
def test_staged_layers(cfg, skip):
    lib()
    E, S = cfg.E, cfg.S
    w = Workload(cfg, gen_device="cpu", extra_rows=2 * E)
    layers = [0, 1, 2, 0]
    ocache = SlotCache.from_state(S, cfg.L, E, w.prefill["slot_key"], w.prefill["slot_ts"],
                                  w.prefill["clock"])
    assert np.array_equal(oes.slot_cache_read_state(w.cache, S, cfg.L, E)["map"], ocache.map)
    maps = [ocache.map[l * E:(l + 1) * E] for l in layers]
    assert any((m >= 0).any() for m in maps), "the pre-fill must leave some experts resident"
    plan = oes.oes_stage_plan_create(w.cache, layers, skip)
    for i, m in enumerate(maps):
        runs, rows = oes.oes_stage_plan_layer(plan, i, E)
        want_runs, want_rows = stage_runs(m, skip)
        assert runs == want_runs and rows == want_rows
    slots_before = w.pool.clone()
    runs_ = [Run(w) for _ in layers]
    oes.moe_layers_forward_staged(plan, w.src, w.pool_all, runs_[0].desc, [r.chunk for r in runs_],
                                  copy_stream=torch.cuda.Stream())
    torch.cuda.synchronize()
    for i, l in enumerate(layers):
        assert int(runs_[i].status.item()) == 0
        s = gpu_stream(w, layer=l)
        assert torch.equal(s.out.view(torch.int16), runs_[i].out.view(torch.int16)), (i, l)
    assert torch.equal(w.pool, slots_before), "resident rows must stay untouched"
    # the oracle over its own pool model: staged rows from the source, the rest from the slots
    pool = w.oracle_pool()
    _copied, reads = staged_pool(pool, S, E, layers, maps, w.source_row, skip)
    last = len(layers) - 1
    b = last % 2
    for e in range(E):
        if reads[last][e] >= S:
            got = w.pool_all[S + b * E + e].cpu().numpy()
            assert np.array_equal(got, w.source_row(layers[last], e)), e
    outs = forward_staged_layers(cfg, w.rin, w.oracle_pool(), S, layers, maps, w.source_row, skip,
                                 block=oes.oes_tile_plan(cfg.T * cfg.k, E))
    for i in (0, 2):
        check_close(runs_[i].out, outs[i]["out"], cfg.wfmt)
    oes.oes_stage_plan_destroy(plan)
    w.close()


def test_staged_plan_refuses_bad_layers():
    lib()
    w = Workload(STAGE_BF16, gen_device="cpu", extra_rows=2 * STAGE_BF16.E)
    with pytest.raises(oes.OesError) as e:
        oes.oes_stage_plan_create(w.cache, [0, 3], True)
    assert e.value.code == oes.OES_ERR_INVALID_ARG
    w.close()
