"""Prefill staging over a sequence of layers.

Test infrastructure only.  vLLM fork PR #51, Details ("Prefill staging"):
one placement readback per step turns each layer's experts without a slot
into maximal contiguous runs; those rows are copied into a whole-layer
staging buffer (two buffers, alternating by layer); experts with a slot are
read from the pool and their rows are never written.  Its test counts the
layers that went through a staging buffer and the rows that moved, checks
that rows already in the pool kept their bytes, and compares the output
with the unstaged read byte for byte.

Readings: with skip_resident off every expert is staged (the whole-layer
stream with next-layer prefetch); an expert's weights come from its slot
when it has one, else from its staging row, so the output equals the
streamed layer's whenever every resident slot holds its source row.
"""
from __future__ import annotations

import numpy as np

from .layer import forward_stream


def stage_runs(map_row: np.ndarray, skip_resident: bool):
    """map_row [E]: slot of each expert of one layer (-1 = none).  Returns
    the maximal ascending runs [e0, e1) of experts to stage and their count."""
    E = map_row.size
    staged = [not (skip_resident and map_row[e] >= 0) for e in range(E)]
    runs = []
    e = 0
    while e < E:
        if staged[e]:
            e0 = e
            while e < E and staged[e]:
                e += 1
            runs.append((e0, e))
        else:
            e += 1
    return runs, sum(staged)


def staged_pool(pool: dict, S: int, E: int, plan_layers, map_rows, source_row, skip_resident,
                first: int = 0):
    """Runs the copies of a staged step on the pool model (slot -> bytes,
    rows S + b*E + e for staging buffer b; the step's layers are the plan's
    layers first, first+1, ...) and returns, per layer, the staged rows and
    the row each expert is read from."""
    reads, copied = [], []
    for i, (layer, m) in enumerate(zip(plan_layers, map_rows), start=first):
        b = i % 2
        runs, n = stage_runs(m, skip_resident)
        for e0, e1 in runs:
            for e in range(e0, e1):
                pool[S + b * E + e] = source_row(layer, e)
        copied.append(n)
        reads.append([int(m[e]) if (skip_resident and m[e] >= 0) else S + b * E + e
                      for e in range(E)])
    return copied, reads


def forward_staged(cfg, router_in, pool: dict, read_rows, block, tokens=None):
    """One staged layer: the streamed layer's computation with expert e's
    row taken from pool[read_rows[e]]."""
    return forward_stream(cfg, router_in, lambda e: pool[read_rows[e]], block, tokens=tokens)


def forward_staged_layers(cfg, router_in, pool: dict, S, layers, map_rows, source_row,
                          skip_resident, block, tokens=None):
    """A staged step in order: layer i is staged into buffer i % 2 (over
    whatever layer i-2 left there) and computed before layer i+1 is staged.
    Returns each layer's forward_staged result."""
    outs = []
    for i, (layer, m) in enumerate(zip(layers, map_rows)):
        _n, reads = staged_pool(pool, S, cfg.E, [layer], [m], source_row, skip_resident,
                                first=i)
        outs.append(forward_staged(cfg, router_in, pool, reads[0], block, tokens=tokens))
    return outs
