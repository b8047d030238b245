"""The chunk's distinct experts as a sorted list of fixed length.

Test infrastructure only.  FreeToken PR #676, Solution: the distinct experts
form a sorted list whose length is fixed in advance, so the host never waits
to learn it; gdevenyi's review comment on the same page dedups the ids
first, which bounds them by num_experts.  Reading: length min(R, E), ascending, padded at the
tail with -1; ids outside [0, E) are not experts and are dropped.
"""
from __future__ import annotations

import numpy as np


def distinct_experts(ids: np.ndarray, E: int):
    flat = [int(v) for v in np.asarray(ids).reshape(-1)]
    seen = sorted(set(v for v in flat if 0 <= v < E))
    n = min(len(flat), E)
    out = np.full(n, -1, dtype=np.int32)
    out[: len(seen)] = seen
    return out, len(seen)
