"""Pins for the oracle's prefill staging (CPU only).

* The hand case in tests/golden/stage_hand.json (vLLM fork PR #51, Details
  and its staging test: both layers go through a buffer, 8 rows move, rows
  already in the pool keep their bytes), with and without skipping resident
  experts.
* Brute force: on random placements the runs are ascending, disjoint,
  maximal, and cover exactly the experts without a slot.
* The staged layer equals the streamed layer when every slot holds its
  source row, and differs when a resident slot is stale (so the oracle
  really reads resident experts from the pool).
"""
import json
import os

import numpy as np
import pytest

from conftest import GOLDEN
from offloaded_expert_slot_gb300.configs import C1, scaled
from offloaded_expert_slot_gb300.inputs import expert_rows, router_inputs
from oracle.layer import forward_stream
from oracle.stage import forward_staged, stage_runs, staged_pool


def test_hand_case():
    g = json.load(open(os.path.join(GOLDEN, "stage_hand.json")))
    E, S = g["E"], g["S"]
    maps = [np.array(m) for m in g["map"]]
    for skip, key in [(True, "skip_resident"), (False, "whole_layer")]:
        want = g[key]
        for i, m in enumerate(maps):
            runs, n = stage_runs(m, skip)
            assert [list(r) for r in runs] == want["runs"][i]
            assert n == want["rows"][i]
        pool = {s: ("slot", s) for s in range(S)}
        before = dict(pool)
        copied, reads = staged_pool(pool, S, E, g["layers"], maps,
                                    lambda l, e: ("src", l, e), skip)
        assert copied == want["rows"] and reads == want["reads"]
        assert all(pool[s] == before[s] for s in range(S))     # resident rows untouched
        for i, (l, m) in enumerate(zip(g["layers"], maps)):
            for e in range(E):
                r = reads[i][e]
                assert pool[r] == (("slot", int(m[e])) if r < S else ("src", l, e))
    assert sum(g["skip_resident"]["rows"]) == 8


@pytest.mark.parametrize("seed", range(40))
def test_runs_cover_exactly_the_non_resident(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 70))
    m = np.where(rng.random(E) < rng.random(), rng.integers(0, 100, E), -1)
    runs, n = stage_runs(m, True)
    covered = [e for a, b in runs for e in range(a, b)]
    assert covered == [e for e in range(E) if m[e] < 0] and n == len(covered)
    for (a0, a1), (b0, b1) in zip(runs, runs[1:]):
        assert a1 < b0                              # disjoint and not adjacent: maximal
    for a, b in runs:
        assert a < b and (a == 0 or m[a - 1] >= 0) and (b == E or m[b] >= 0)
    assert stage_runs(m, False) == ([(0, E)], E)


def test_staged_layer_equals_stream_and_reads_the_pool():
    cfg = scaled(C1, name="stage_tiny", S=8, L=2)
    rin = router_inputs(cfg)
    rows = {l: expert_rows(cfg, l, list(range(cfg.E)), device="cpu") for l in range(cfg.L)}
    src = lambda l, e: rows[l][e]
    m = np.array([-1, 0, 3, -1, -1, 5, -1, -1])
    pool = {0: src(1, 1), 3: src(1, 2), 5: src(1, 5)}
    _copied, reads = staged_pool(pool, cfg.S, cfg.E, [1], [m], src, True)
    got = forward_staged(cfg, rin, pool, reads[0], block=16)
    want = forward_stream(cfg, rin, lambda e: src(1, e), block=16)
    assert np.array_equal(got["out"], want["out"])
    pool[3] = src(0, 2)                                   # stale resident slot
    bad = forward_staged(cfg, rin, pool, reads[0], block=16)
    assert not np.array_equal(bad["out"], want["out"])


def test_staged_sequence_reuses_buffers_in_order():
    """Layers 1, 0, 1 through two buffers: the third layer overwrites the
    first's buffer, and each layer still reads its own rows."""
    from oracle.stage import forward_staged_layers
    cfg = scaled(C1, name="stage_tiny", S=8, L=2)
    rin = router_inputs(cfg)
    rows = {l: expert_rows(cfg, l, list(range(cfg.E)), device="cpu") for l in range(cfg.L)}
    src = lambda l, e: rows[l][e]
    maps = [np.full(cfg.E, -1)] * 3
    outs = forward_staged_layers(cfg, rin, {}, cfg.S, [1, 0, 1], maps, src, True, block=16)
    for o, l in zip(outs, [1, 0, 1]):
        want = forward_stream(cfg, rin, lambda e: src(l, e), block=16)
        assert np.array_equal(o["out"], want["out"])
    assert not np.array_equal(outs[0]["out"], outs[1]["out"])
