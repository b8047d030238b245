"""The N>1 bench path: independent replicas, one per rank, no data-path
collective; the job's step time is the slowest rank's and its throughput
counts every rank's tokens.  Run as two gloo ranks on the CPU.

Each rank runs the whole slot path of the oracle (routing, distinct experts,
the LRU queries with their miss copies into its own pool model, align,
expert MLP, combine) on its own replica workload, with its own cache, and
the only collective is the max of the step times.  Its tables, miss lists
and output must equal a single-process run of the same replica: nothing
one rank does reaches the other."""
import os
import socket
import time

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _small():
    import sys
    sys.path.insert(0, ROOT)
    from offloaded_expert_slot_gb300.configs import C2, scaled
    return scaled(C2, name="replica_small", T=12, k=4, E=16, H=128, I=64, S=40, L=2, prefill=20,
                  query_width=8)


def _replica(cfg):
    """One replica's slot path on the oracle: everything it produces."""
    import sys
    sys.path.insert(0, ROOT)
    from offloaded_expert_slot_gb300.inputs import (empty_slot_row, expert_layer_rows,
                                                    pool_prefill, router_inputs)
    from oracle.layer import forward_slots
    from oracle.slot_cache import SlotCache
    rows = [expert_layer_rows(cfg, l).numpy() for l in range(cfg.L)]
    st = pool_prefill(cfg)
    cache = SlotCache.from_state(cfg.S, cfg.L, cfg.E, st["slot_key"], st["slot_ts"], st["clock"])
    empty = empty_slot_row(cfg)
    pool = {s: (rows[k // cfg.E][k % cfg.E] if k >= 0 else empty)
            for s, k in enumerate(st["slot_key"])}
    o = forward_slots(cfg, router_inputs(cfg), lambda l, e: rows[l][e], cache, pool, block=16)
    misses = np.array([m for q in o["queries"] for m in q["misses"]], dtype=np.int64).reshape(-1, 3)
    pool_keys = np.array([int(cache.slot_key[s]) for s in range(cfg.S)])
    return {"ids": o["ids"], "w": o["w"], "distinct": o["distinct"], "misses": misses,
            "map": cache.map.copy(), "slot_key": cache.slot_key.copy(),
            "slot_ts": cache.slot_ts.copy(), "sorted_ids": o["sorted_ids"],
            "block_expert": o["block_expert"], "out": o["out"], "pool_keys": pool_keys,
            "ok": np.array([o["ok"]])}


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    cfg = bench.replica_config(_small(), rank)
    t0 = time.perf_counter()
    res = _replica(cfg)
    ms = (time.perf_counter() - t0) * 1e3
    ms_max = bench.reduce_max(ms, dist, "cpu")
    value = bench.job_value(cfg.T, world, ms_max)
    dist.barrier()
    out[rank] = (res, ms, ms_max, value, cfg.seed)
    dist.destroy_process_group()


def test_two_rank_replicas_are_independent_and_take_the_slowest_rank():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    base = _small()
    seeds = [out[r][4] for r in range(world)]
    assert seeds[0] == base.seed and seeds[1] != seeds[0]
    for r in range(world):
        res, ms, ms_max, value, _ = out[r]
        alone = _replica(bench.replica_config(base, r))
        assert res["ok"][0]
        for key, want in alone.items():
            assert np.array_equal(res[key], want), (r, key)
        assert ms_max == max(out[i][1] for i in range(world))
        assert value == pytest.approx(base.T * world / (ms_max / 1e3))
    # the two replicas worked on different chunks
    assert not np.array_equal(out[0][0]["ids"], out[1][0]["ids"])


def test_single_process_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(2.5, None, "cpu") == 2.5
    assert bench.job_value(32, 1, 2.0) == pytest.approx(16000.0)
    assert bench.replica_config(_small(), 0) is _small() or bench.replica_config(_small(), 0) == _small()
