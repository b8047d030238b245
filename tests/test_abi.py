"""The C-ABI library builds, loads and exports every call include/oes.h
declares; host-side argument checks work without a GPU (CPU only)."""
import os
import re

import pytest

from conftest import ROOT
from offloaded_expert_slot_gb300 import build, oes


@pytest.fixture(scope="module")
def lib():
    build.build()
    return oes.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "oes.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "for")))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(oes._SIGS)


def test_host_argument_checks(lib):
    with pytest.raises(oes.OesError) as e:
        oes.moe_route_topk(0, 4, 8, 2, 0, 0, stream=0)
    assert e.value.code == oes.OES_ERR_INVALID_ARG
    with pytest.raises(oes.OesError) as e:
        oes.moe_route_topk(16, 4, 8, 9, 16, 16, stream=0)     # k > E
    assert e.value.code == oes.OES_ERR_INVALID_ARG
    with pytest.raises(oes.OesError) as e:
        oes.moe_route_topk(16, 4, 8, 2, 16, 16, stream=0, dtype=7)   # unknown logits type
    assert e.value.code == oes.OES_ERR_INVALID_ARG
    with pytest.raises(oes.OesError) as e:
        oes.slot_cache_create(0, 1, 8)
    assert e.value.code == oes.OES_ERR_INVALID_ARG
    with pytest.raises(oes.OesError) as e:
        oes.slot_cache_create(oes.OES_MAX_SLOTS + 1, 1, 8)
    assert e.value.code == oes.OES_ERR_INVALID_ARG
    with pytest.raises(oes.OesError) as e:
        oes.moe_align_block_size(16, 4, 0, 16, 1, 16, 16, 16, 0, 16, 1 << 20, stream=0)   # E = 0
    assert e.value.code == oes.OES_ERR_INVALID_ARG
    with pytest.raises(oes.OesError) as e:
        oes.slot_cache_ensure(0, 0, 16, 4, 0, 16, 16, 16, stream=0)   # null cache
    assert e.value.code == oes.OES_ERR_INVALID_ARG


def test_tile_plan_uses_the_layers_expert_count(lib):
    """FreeToken PR #676, Solution and Tests: tiles follow routes per expert
    of the layer, never of the slot pool.  At 600 tokens x
    top-10 the layer's 512 experts get 11.7 routes each (blocks of 128 routes,
    token-major kernel); sizing by the 1100 slots would give 5.5 (blocks of
    16, weight-major kernel)."""
    assert oes.oes_tile_plan(600 * 10, 512) == 128
    assert oes.oes_tile_plan(600 * 10, 1100) == 16
    assert oes.oes_tile_plan(4096 * 10, 512) == 128
    assert oes.oes_tile_plan(32 * 10, 512) == 16
    assert oes.oes_tile_plan(200 * 10, 512) == 16
    assert oes.oes_tile_plan(16 * 2, 8) == 16
    for R, E, want in [(8 * 512, 512, 16), (8 * 512 + 1, 512, 128), (0, 5, 16)]:
        assert oes.oes_tile_plan(R, E) == want


def test_align_capacity_macro_matches_the_oracle():
    from oracle.align import align_capacity
    for R, E, B in [(0, 5, 4), (1, 1, 1), (10, 3, 8), (40960, 512, 128), (65536, 2100, 64)]:
        assert oes.align_capacity(R, E, B) == align_capacity(R, E, B)


def test_demand_token_dispatch_rule(lib):
    """The page's threshold examples (tests/golden/demand_dispatch.json)."""
    import json
    from conftest import GOLDEN
    for c in json.load(open(os.path.join(GOLDEN, "demand_dispatch.json")))["cases"]:
        assert oes.oes_takes_slot_path(c["T"], c["k"], c["E"], c["S"], c["N"]) == c["slots"], c


def test_logits_type_follows_the_array():
    """The binding names the logits type from the array: fp32, or bf16 given as
    bf16 or as its 16-bit patterns; any other type is refused before a call."""
    import numpy as np
    import torch
    assert oes._logits_type(np.zeros(2, np.float32)) == oes.OES_LOGITS_F32
    assert oes._logits_type(torch.zeros(2)) == oes.OES_LOGITS_F32
    for a in (np.zeros(2, np.uint16), torch.zeros(2, dtype=torch.bfloat16),
              torch.zeros(2, dtype=torch.int16)):
        assert oes._logits_type(a) == oes.OES_LOGITS_BF16
    for a in (torch.zeros(2, dtype=torch.float16), np.zeros(2, np.float64)):
        with pytest.raises(TypeError):
            oes._logits_type(a)


def test_null_handles_destroy_as_no_ops(lib):
    oes.slot_cache_destroy(None)
    with pytest.raises(oes.OesError):
        oes.slot_cache_reset(None, stream=0)
    oes.oes_expert_source_destroy(None)
    oes.oes_stage_plan_destroy(None)


def _invalid(fn, *args, **kw):
    with pytest.raises(oes.OesError) as e:
        fn(*args, **kw)
    assert e.value.code == oes.OES_ERR_INVALID_ARG, e.value
    return str(e.value)


def test_handle_and_layer_argument_checks(lib):
    """Checks that the library takes on the host, before any device work: the
    addresses below are never dereferenced."""
    A = 1 << 20                                    # a fake, 256-byte aligned address
    # slot cache: L * E must stay below 2^31, E within OES_MAX_EXPERTS
    _invalid(oes.slot_cache_create, 16, 1 << 20, 4096)
    _invalid(oes.slot_cache_create, 16, 1, oes.OES_MAX_EXPERTS + 1)
    _invalid(oes.slot_cache_create, 16, 0, 8)
    # expert source: row size a positive multiple of 16, bases non-null and aligned
    _invalid(oes.oes_expert_source_create, [A, A], 8, 24)
    _invalid(oes.oes_expert_source_create, [A, A], 8, 0)
    msg = _invalid(oes.oes_expert_source_create, [A, A + 8], 8, 64)
    assert "layer 1" in msg
    _invalid(oes.oes_expert_source_create, [A, 0], 8, 64)
    # stage plan and its per-layer query need a plan
    _invalid(oes.oes_stage_plan_create, None, [0], 0, stream=0)
    _invalid(oes.oes_stage_plan_layer, None, 0, 8)
    # a whole-layer chunk is validated before the cache, source or pool
    desc = oes.layer_desc(8, 64, 32, oes.OES_WFMT_BF16)
    need = oes.moe_layer_workspace_size(desc, 4, 2)
    assert need > 0 and need % 256 == 0
    ok = dict(x=A, T=4, k=2, out=A, status=A, workspace=A, workspace_bytes=need, logits=A)
    for bad in [dict(workspace_bytes=need - 1), dict(workspace=A + 16), dict(k=9), dict(k=0),
                dict(T=-1), dict(x=None), dict(logits=None), dict(out=None)]:
        ch = oes.chunk(**{**ok, **bad})
        msg = _invalid(oes.moe_layer_forward_slots, A, A, A, 0, desc, ch, False, stream=0)
        assert "layer forward" in msg, bad
        _invalid(oes.moe_layer_forward_stream, A, A, 0, desc, ch, copy_stream=0,
                 compute_stream=0)
    ch = oes.chunk(**ok)
    msg = _invalid(oes.moe_layer_forward_slots, None, A, A, 0, desc, ch, False, stream=0)
    assert "moe_layer_forward_slots" in msg
    msg = _invalid(oes.moe_layer_forward_stream, None, A, 0, desc, ch, copy_stream=0,
                   compute_stream=0)
    assert "moe_layer_forward_stream" in msg
    _invalid(oes.moe_layers_forward_staged, None, A, A, desc, [ch], copy_stream=0,
             compute_stream=0)
