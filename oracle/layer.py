"""The whole MoE layer forward: over the slot cache, and streamed.

Test infrastructure only.  FreeToken PR #676, Solution: a short prefill
chunk brings only its routed experts into the slot cache, the way decode
does, then reuses the decode GEMM with each expert read at its slot, and
must give exactly the streamed layer's bytes; the streamed path moves all of
the layer's experts (Problem).  Slot path, in the pages' order:
route -> distinct experts -> queries of at most `query_width` keys, each
query ensured and its misses copied before the next -> expert->slot remap
(vLLM fork PR #48, What: physical-row remap) -> align -> expert MLP reading
each expert's weights from the pool at its slot -> combine.

The pool is modelled as a dict slot -> row bytes; a copy puts the host
source's row of the missing key into its slot.
"""
from __future__ import annotations

import numpy as np

from .align import moe_align_block_size
from .distinct import distinct_experts
from .expert_mlp import combine, expert_weights, input_scales, swiglu_expert, swiglu_expert_w4a4
from .numerics import bf16_to_f64
from .router import gate_logits, route_topk
from .slot_cache import OK


def route(router_in: dict, k: int):
    logits = router_in.get("logits")
    if logits is None:
        logits = gate_logits(router_in["x"], router_in["gate"])
    ids, w = route_topk(logits, k)
    return logits, ids, w


def _wfmt(cfg) -> str:
    return "nvfp4_w4a4" if getattr(cfg, "w4a4", False) else cfg.wfmt


def layer_act_scales(layer_row, E, H, I):
    """W4A4 activation scales of a layer: the maximum of its experts' w13
    and w2 input scales, read from the layer's own rows (FreeToken PR #676,
    Solution and Tests: the layer's scales, not other slots')."""
    s = [input_scales(layer_row(e), H, I) for e in range(E)]
    return max(v[0] for v in s), max(v[1] for v in s)


def expert_outputs(x_bits, ids, row_of_expert, wfmt, H, I, tokens=None, act=None):
    """y [R, H] fp64 for the routes of `tokens` (all tokens when None); other
    rows are NaN.  row_of_expert(e) -> that expert's row bytes.  act: the
    (a13, a2) activation scales of a W4A4 layer."""
    T, k = ids.shape
    x = bf16_to_f64(x_bits)
    y = np.full((T * k, H), np.nan, dtype=np.float64)
    toks = np.arange(T) if tokens is None else np.asarray(tokens)
    routes = (toks[:, None] * k + np.arange(k)[None, :]).reshape(-1)
    by_expert = {}
    for r in routes:
        by_expert.setdefault(int(ids.reshape(-1)[r]), []).append(int(r))
    w4a4 = wfmt == "nvfp4_w4a4"
    for e, rs in sorted(by_expert.items()):
        w13, w2 = expert_weights(row_of_expert(e), "nvfp4" if w4a4 else wfmt, H, I)
        rs = np.array(rs)
        if w4a4:
            y[rs] = swiglu_expert_w4a4(x[rs // k], w13, w2, act[0], act[1])
        else:
            y[rs] = swiglu_expert(x[rs // k], w13, w2)
    return y


def forward_slots(cfg, router_in, source_row, cache, pool, block, layer=None,
                  record_stats=False, tokens=None, query_width=None, tag=0):
    """source_row(layer, e) -> host source row bytes; cache: SlotCache;
    pool: dict slot -> row bytes (updated by the copies).

    The pool must hold all of the chunk's experts at once (FreeToken PR
    #676, the author's reply; gdevenyi fork PR #68 streams a layer that
    needs too much of the cache).  The bound known before routing is min(R, E): a
    chunk with min(R, E) > S is refused here and takes the streamed path.
    """
    layer = cfg.layer if layer is None else layer
    W = query_width or cfg.query_width
    E, k = cfg.E, cfg.k
    if min(cfg.T * k, E) > cfg.S:
        return {"ok": False, "capacity": True}
    logits, ids, w = route(router_in, k)
    distinct, D = distinct_experts(ids, E)
    queries = []
    for q0 in range(0, distinct.size, W):
        part = distinct[q0:q0 + W]
        keys = [layer * E + int(e) if e >= 0 else -1 for e in part]
        status, misses = cache.ensure(keys, record_stats=record_stats, tag=tag)
        for key, slot, _old in misses:
            pool[slot] = source_row(key // E, key % E)
        queries.append({"keys": keys, "status": status, "misses": misses})
    e2s = cache.map[layer * E:(layer + 1) * E].copy()
    sorted_ids, block_expert, n_post_pad, _bad = moe_align_block_size(ids.reshape(-1), E, block)
    act = (layer_act_scales(lambda e: source_row(layer, e), E, cfg.H, cfg.I)
           if getattr(cfg, "w4a4", False) else None)
    y = expert_outputs(router_in["x"], ids, lambda e: pool[int(e2s[e])], _wfmt(cfg), cfg.H, cfg.I,
                       tokens=tokens, act=act)
    out = combine(np.nan_to_num(y), w, cfg.T, k)
    return {"logits": logits, "ids": ids, "w": w, "distinct": distinct, "D": D,
            "queries": queries, "e2s": e2s, "sorted_ids": sorted_ids,
            "block_expert": block_expert, "n_post_pad": n_post_pad, "y": y, "out": out,
            "ok": all(q["status"] == OK for q in queries), "capacity": False}


def forward_stream(cfg, router_in, layer_rows, block, tokens=None):
    """layer_rows(e) -> row bytes of expert e of the streamed layer."""
    E, k = cfg.E, cfg.k
    logits, ids, w = route(router_in, k)
    sorted_ids, block_expert, n_post_pad, _bad = moe_align_block_size(ids.reshape(-1), E, block)
    act = layer_act_scales(layer_rows, E, cfg.H, cfg.I) if getattr(cfg, "w4a4", False) else None
    y = expert_outputs(router_in["x"], ids, layer_rows, _wfmt(cfg), cfg.H, cfg.I, tokens=tokens,
                       act=act)
    out = combine(np.nan_to_num(y), w, cfg.T, k)
    return {"ids": ids, "w": w, "sorted_ids": sorted_ids, "block_expert": block_expert,
            "n_post_pad": n_post_pad, "y": y, "out": out}
