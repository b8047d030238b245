"""Runs the slot path of one workload for a few steps, for a profiler.

    python -m offloaded_expert_slot_gb300.profile_case [--config NAME]
        [--slots S --prefill P] [--tokens T] [--steps N] [--warm]

Each step restores the cache tables to the workload's seeded pre-fill and
runs moe_layer_forward_slots on the default stream, as bench.py's timed
step does.  --warm skips the restore: from the second step on every expert
of the chunk is resident, and the GEMM over the hits covers the whole chunk
in one GEMM1 + GEMM2 launch pair (the first two grouped-GEMM launches of
that step).  --slots / --prefill shrink the pool (a smaller case with the
same kernels and shapes, for multi-pass captures).  Exits non-zero if the
device status is not 0.
"""
from __future__ import annotations

import argparse
import sys

import numpy as np


def main() -> int:
    import torch

    from . import build, oes
    from .configs import CONFIGS, scaled
    from .inputs import (empty_slot_row, expert_layer_rows, n_source_buffers, pool_prefill,
                         router_inputs, source_layer_index)

    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="c2_decode_width", choices=sorted(CONFIGS))
    ap.add_argument("--slots", type=int, default=0)
    ap.add_argument("--prefill", type=int, default=-1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warm", action="store_true")
    ap.add_argument("--tokens", type=int, default=0)
    a = ap.parse_args()
    cfg = CONFIGS[a.config]
    if a.slots:
        cfg = scaled(cfg, S=a.slots)
    if a.prefill >= 0:
        cfg = scaled(cfg, prefill=a.prefill)
    if a.tokens:
        cfg = scaled(cfg, T=a.tokens)
    build.build()
    oes.load()
    rb, E = cfg.row_bytes, cfg.E
    srcs = []
    for l in range(n_source_buffers(cfg)):
        buf = torch.empty((E, rb), dtype=torch.uint8, pin_memory=True)
        expert_layer_rows(cfg, l, device="cuda", out=buf)
        srcs.append(buf)
    src = oes.oes_expert_source_create([srcs[source_layer_index(cfg, l)] for l in range(cfg.L)],
                                       E, rb)
    pool = torch.empty((cfg.S, rb), dtype=torch.uint8, device="cuda")
    cache = oes.slot_cache_create(cfg.S, cfg.L, E)
    st = pool_prefill(cfg)
    oes.slot_cache_load_state(cache, st["slot_key"], st["slot_ts"], st["clock"])
    pool[:] = torch.from_numpy(empty_slot_row(cfg)).cuda()
    for s in np.nonzero(st["slot_key"] >= 0)[0]:
        key = int(st["slot_key"][s])
        pool[int(s)].copy_(srcs[source_layer_index(cfg, key // E)][key % E])
    snap = torch.empty(oes.slot_cache_state_bytes(cache), dtype=torch.uint8, device="cuda")
    oes.slot_cache_snapshot(cache, snap)
    rin = router_inputs(cfg)
    x = torch.from_numpy(rin["x"].view(np.int16)).cuda()
    logits = torch.from_numpy(rin["logits"]).cuda() if rin["logits"] is not None else None
    gate = torch.from_numpy(rin["gate"].view(np.int16)).cuda() if rin["gate"] is not None else None
    wfmt = oes.OES_WFMT_BF16 if cfg.wfmt == "bf16" else oes.OES_WFMT_NVFP4
    desc = oes.layer_desc(E, cfg.H, cfg.I, wfmt)
    wsb = oes.moe_layer_workspace_size(desc, cfg.T, cfg.k)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ch = oes.chunk(x, cfg.T, cfg.k, out, status, ws, wsb, logits=logits, gate=gate)
    torch.cuda.synchronize()
    for _ in range(a.steps):
        if not a.warm:
            oes.slot_cache_restore(cache, snap)
        oes.moe_layer_forward_slots(cache, src, pool, cfg.layer, desc, ch, 0)
    torch.cuda.synchronize()
    code = int(status.item())
    oes.slot_cache_destroy(cache)
    oes.oes_expert_source_destroy(src)
    print(f"{cfg.name}: S={cfg.S} prefill={cfg.prefill} steps={a.steps} warm={a.warm} "
          f"status={code}")
    return 0 if code == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
