"""moe_align_block_size as a stable counting sort of routes by expert.

Test infrastructure only.  Sources: FreeToken PR #676, Solution and Tests
(the align must be right past 1024 experts, with each route placed exactly
once and only in a block of its own expert), gdevenyi's review comment there
(sgl_kernel's single-block align breaks once num_experts + 1 exceeds 1024
threads), vLLM fork PR #48, What
(logical alignment with ignore_invalid_experts, then a physical-row remap).

Input: ids [R] (route r = t*k + j), E experts, block size B.
Output:
  sorted_ids [cap]: for each expert e in ascending order, its routes in
      ascending route id, then padding up to a multiple of B; the padding
      value is R; every entry past the last block is R too;
  block_expert [cap/B]: the expert of each block, -1 past the last block;
  n_post_pad: the number of used entries (a multiple of B).
Experts with no route get no block.  ids outside [0, E) are skipped; when
ignore_invalid is false their presence is also reported (bad = True).
cap = R + min(E, R) * (B - 1), rounded up to a multiple of B: no routing can
need more.
"""
from __future__ import annotations

import numpy as np


def align_capacity(R: int, E: int, B: int) -> int:
    c = R + min(E, R) * (B - 1)
    return (c + B - 1) // B * B


def moe_align_block_size(ids: np.ndarray, E: int, B: int, ignore_invalid: bool = True):
    ids = np.asarray(ids, dtype=np.int64).reshape(-1)
    R = ids.size
    cap = align_capacity(R, E, B)
    cnt = [0] * E
    bad = False
    for v in ids:
        if 0 <= v < E:
            cnt[int(v)] += 1
        else:
            bad = True
    padded = [(c + B - 1) // B * B for c in cnt]
    off = [0] * E
    run = 0
    for e in range(E):
        off[e] = run
        run += padded[e]
    n_post_pad = run
    sorted_ids = np.full(cap, R, dtype=np.int32)
    block_expert = np.full(cap // B, -1, dtype=np.int32)
    fill = list(off)
    for r in range(R):
        v = int(ids[r])
        if 0 <= v < E:
            sorted_ids[fill[v]] = r
            fill[v] += 1
    for e in range(E):
        for b in range(off[e] // B, (off[e] + padded[e]) // B):
            block_expert[b] = e
    return sorted_ids, block_expert, n_post_pad, (bad and not ignore_invalid)
