"""ctypes binding of liboes.so: argument marshalling only.

Every function here has the name of the C call it forwards to (include/oes.h)
and does nothing but turn tensors / ints into raw pointers and sizes, call the
library, and raise OesError on a non-zero return code.  Every step of the
path runs in the library's CUDA kernels; there is no other implementation,
and loading fails loudly when the library has not been built.

Tensors are torch tensors (device memory unless a call says "mapped" or
"host"); a plain int is taken as a raw address.  `stream` is a
torch.cuda.Stream, a raw cudaStream_t as int, or None for torch's current
stream.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

OES_OK, OES_ERR_INVALID_ARG, OES_ERR_UNSUPPORTED, OES_ERR_CUDA, OES_ERR_CAPACITY = range(5)
OES_DEV_CAPACITY, OES_DEV_BAD_ID, OES_DEV_TIMEOUT = 1, 2, 4
OES_WFMT_BF16, OES_WFMT_NVFP4, OES_WFMT_NVFP4_W4A4 = 0, 1, 2
OES_LOGITS_F32, OES_LOGITS_BF16 = 0, 1
OES_POLICY_LRU, OES_POLICY_LRFU = 0, 1
OES_LRFU_MAX_K = 18
OES_QUERY_MAX = 128
OES_MAX_TOPK = 32
OES_MAX_EXPERTS = 4096
OES_MAX_SLOTS = 8192

_ERR_NAMES = {1: "OES_ERR_INVALID_ARG", 2: "OES_ERR_UNSUPPORTED", 3: "OES_ERR_CUDA",
              4: "OES_ERR_CAPACITY"}


class OesError(RuntimeError):
    def __init__(self, code: int, func: str, msg: str):
        super().__init__(f"{func}: {_ERR_NAMES.get(code, code)}: {msg}")
        self.code = code


def align_capacity(R: int, E: int, B: int) -> int:
    """OES_ALIGN_CAPACITY from the header."""
    c = R + min(E, R) * (B - 1)
    return (c + B - 1) // B * B


class RoutedExperts(C.Structure):
    _fields_ = [("layer", C.c_int), ("E", C.c_int), ("e2s", C.c_void_p), ("wfmt", C.c_int),
                ("pool", C.c_void_p), ("row_bytes", C.c_int64), ("S", C.c_int), ("H", C.c_int),
                ("I", C.c_int), ("input_scale13", C.c_void_p), ("input_scale2", C.c_void_p)]


class Chunk(C.Structure):
    _fields_ = [("logits", C.c_void_p), ("gate", C.c_void_p), ("x", C.c_void_p), ("T", C.c_int),
                ("k", C.c_int), ("out", C.c_void_p), ("status", C.c_void_p),
                ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t)]


class LayerDesc(C.Structure):
    _fields_ = [("E", C.c_int), ("H", C.c_int), ("I", C.c_int), ("wfmt", C.c_int),
                ("input_scale13", C.c_void_p), ("input_scale2", C.c_void_p)]


_lib = None
_vp, _i, _i64, _sz = C.c_void_p, C.c_int, C.c_int64, C.c_size_t
_SIGS = {
    "oes_last_error": (C.c_char_p, []),
    "moe_gate_logits": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp]),
    "moe_route_topk": (_i, [_vp, _i, _i, _i, _i, _vp, _vp, _vp]),
    "moe_distinct_experts": (_i, [_vp, _i, _i, _vp, _vp, _vp]),
    "slot_cache_create": (_i, [_i, _i, _i, C.POINTER(_vp)]),
    "slot_cache_destroy": (_i, [_vp]),
    "slot_cache_reset": (_i, [_vp, _vp]),
    "slot_cache_load_state": (_i, [_vp, _vp, _vp, _i64]),
    "slot_cache_read_state": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "slot_cache_layer_map": (_i, [_vp, _i, C.POINTER(_vp)]),
    "slot_cache_state_bytes": (_sz, [_vp]),
    "slot_cache_snapshot": (_i, [_vp, _vp, _vp]),
    "slot_cache_restore": (_i, [_vp, _vp, _vp]),
    "slot_cache_ensure": (_i, [_vp, _i, _vp, _i, _i, _vp, _vp, _vp, _vp]),
    "oes_expert_source_create": (_i, [_vp, _i, _i, _i64, C.POINTER(_vp)]),
    "oes_expert_source_destroy": (_i, [_vp]),
    "slot_cache_copy_misses": (_i, [_vp, _vp, _i, _vp, _vp, _i, _vp, _vp]),
    "oes_copy_layer": (_i, [_vp, _i, _vp, _vp]),
    "moe_align_workspace_size": (_sz, [_i, _i, _i]),
    "moe_align_block_size": (_i, [_vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_align_block_size_noalloc": (_i, [_vp, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp]),
    "oes_tile_plan": (_i, [_i, _i, C.POINTER(_i)]),
    "moe_grouped_gemm_workspace_size": (_sz, [C.POINTER(RoutedExperts), _i, _i]),
    "moe_grouped_gemm_slots": (_i, [C.POINTER(RoutedExperts), _vp, _i, _i, _vp, _vp, _vp, _vp, _vp,
                                    _i, _vp, _sz, _vp, _vp, _vp]),
    "moe_layer_workspace_size": (_sz, [C.POINTER(LayerDesc), _i, _i]),
    "moe_layer_workspace_views": (_i, [C.POINTER(LayerDesc), _i, _i, _vp] + [C.POINTER(_vp)] * 7),
    "moe_layer_forward_slots": (_i, [_vp, _vp, _vp, _i, C.POINTER(LayerDesc), C.POINTER(Chunk), _i,
                                     _vp]),
    "moe_layer_forward_stream": (_i, [_vp, _vp, _i, C.POINTER(LayerDesc), C.POINTER(Chunk), _vp,
                                      _vp]),
    "oes_takes_slot_path": (_i, [_i, _i, _i, _i, _i]),
    "slot_cache_ensure_tagged": (_i, [_vp, _i, _vp, _i, _i, C.c_int32, _vp, _vp, _vp, _vp]),
    "slot_cache_set_policy": (_i, [_vp, _i, _i]),
    "slot_cache_read_lrfu": (_i, [_vp, _vp, _vp, _vp]),
    "moe_grouped_gemm_workspace_views": (_i, [C.POINTER(RoutedExperts), _i, _i, _vp, C.POINTER(_vp),
                                              C.POINTER(_vp), C.POINTER(_vp)]),
    "oes_stage_plan_create": (_i, [_vp, C.POINTER(_i), _i, _i, _vp, C.POINTER(_vp)]),
    "oes_stage_plan_destroy": (_i, [_vp]),
    "oes_stage_plan_layer": (_i, [_vp, _i, C.POINTER(_i), _vp, C.POINTER(_i)]),
    "moe_layers_forward_staged": (_i, [_vp, _vp, _vp, C.POINTER(LayerDesc), C.POINTER(Chunk), _vp,
                                       _vp]),
    "moe_layer_forward": (_i, [_vp, _vp, _vp, _vp, _i, C.POINTER(LayerDesc), C.POINTER(Chunk), _i,
                               _i, _vp, _vp, C.POINTER(_i)]),
}


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load liboes.so; raises if it is missing (build it with build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise OSError(f"liboes.so is not built ({path}); run offloaded_expert_slot_gb300.build")
        _build.build()
    lib = C.CDLL(path)
    for name, (res, args) in _SIGS.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int, func: str):
    if rc != OES_OK:
        raise OesError(rc, func, (load().oes_last_error() or b"").decode())


def _call(name, *args):
    rc = getattr(load(), name)(*args)
    _check(rc, name)


# ------------------------------------------------------------------- route
def moe_gate_logits(x, gate, T, H, E, logits, stream=None):
    _call("moe_gate_logits", _ptr(x), _ptr(gate), T, H, E, _ptr(logits), _stream(stream))


def _logits_type(logits) -> int:
    """fp32 arrays are fp32 logits; bf16 arrays and 16-bit integer arrays (bf16
    bit patterns) are bf16; a raw address is fp32 unless dtype says otherwise."""
    if logits is None or isinstance(logits, int):
        return OES_LOGITS_F32
    name = str(getattr(logits, "dtype", "")).replace("torch.", "")
    if name == "float32":
        return OES_LOGITS_F32
    if name in ("bfloat16", "int16", "uint16"):
        return OES_LOGITS_BF16
    raise TypeError(f"moe_route_topk: logits of dtype {name!r}; expected fp32 or bf16 (bit patterns)")


def moe_route_topk(logits, T, E, k, ids, weights, stream=None, dtype=None):
    """dtype: OES_LOGITS_*, or None to take it from the logits array."""
    if dtype is None:
        dtype = _logits_type(logits)
    _call("moe_route_topk", _ptr(logits), dtype, T, E, k, _ptr(ids), _ptr(weights),
          _stream(stream))


def moe_distinct_experts(ids, R, E, distinct, d_count, stream=None):
    _call("moe_distinct_experts", _ptr(ids), R, E, _ptr(distinct), _ptr(d_count), _stream(stream))


# -------------------------------------------------------------- slot cache
def slot_cache_create(S, L, E) -> int:
    h = C.c_void_p()
    _call("slot_cache_create", S, L, E, C.byref(h))
    return h.value


def slot_cache_destroy(cache):
    _call("slot_cache_destroy", cache)


def slot_cache_reset(cache, stream=None):
    _call("slot_cache_reset", cache, _stream(stream))


def slot_cache_load_state(cache, slot_key, slot_ts, clock):
    sk = np.ascontiguousarray(slot_key, dtype=np.int32)
    st = np.ascontiguousarray(slot_ts, dtype=np.int64)
    _call("slot_cache_load_state", cache, sk.ctypes.data, st.ctypes.data, int(clock))


def slot_cache_read_state(cache, S, L, E, stream=None) -> dict:
    m = np.empty(L * E, np.int32)
    sk = np.empty(S, np.int32)
    st = np.empty(S, np.int64)
    clock = np.zeros(1, np.int64)
    ctr = np.zeros(3, np.int64)
    df = np.empty(L * E, np.int64)
    _call("slot_cache_read_state", cache, m.ctypes.data, sk.ctypes.data, st.ctypes.data,
          clock.ctypes.data, ctr.ctypes.data, df.ctypes.data, _stream(stream))
    return {"map": m, "slot_key": sk, "slot_ts": st, "clock": int(clock[0]),
            "hits": int(ctr[0]), "misses": int(ctr[1]), "evictions": int(ctr[2]), "decode_freq": df}


def slot_cache_state_bytes(cache) -> int:
    return int(load().slot_cache_state_bytes(cache))


def slot_cache_snapshot(cache, dst, stream=None):
    _call("slot_cache_snapshot", cache, _ptr(dst), _stream(stream))


def slot_cache_restore(cache, src, stream=None):
    _call("slot_cache_restore", cache, _ptr(src), _stream(stream))


def slot_cache_layer_map(cache, layer) -> int:
    p = C.c_void_p()
    _call("slot_cache_layer_map", cache, layer, C.byref(p))
    return p.value


def slot_cache_ensure(cache, layer, experts, n, record_stats, miss, n_miss, status, stream=None):
    _call("slot_cache_ensure", cache, layer, _ptr(experts), n, int(bool(record_stats)), _ptr(miss),
          _ptr(n_miss), _ptr(status), _stream(stream))


def oes_expert_source_create(layer_bases, E, row_bytes) -> int:
    arr = (C.c_void_p * len(layer_bases))(*[_ptr(b) for b in layer_bases])
    h = C.c_void_p()
    _call("oes_expert_source_create", arr, len(layer_bases), E, row_bytes, C.byref(h))
    return h.value


def oes_expert_source_destroy(src):
    _call("oes_expert_source_destroy", src)


def slot_cache_copy_misses(src, pool, S, miss, n_miss, max_misses, status, stream=None):
    _call("slot_cache_copy_misses", src, _ptr(pool), S, _ptr(miss), _ptr(n_miss), max_misses,
          _ptr(status), _stream(stream))


def oes_copy_layer(src, layer, dst, stream=None):
    _call("oes_copy_layer", src, layer, _ptr(dst), _stream(stream))


# ------------------------------------------------------------------- align
def moe_align_workspace_size(R, E, B) -> int:
    return int(load().moe_align_workspace_size(R, E, B))


def moe_align_block_size(ids, R, E, B, ignore_invalid, sorted_ids, block_expert, n_post_pad,
                         status, workspace, workspace_bytes, stream=None):
    _call("moe_align_block_size", _ptr(ids), R, E, B, int(bool(ignore_invalid)), _ptr(sorted_ids),
          _ptr(block_expert), _ptr(n_post_pad), _ptr(status), _ptr(workspace), workspace_bytes,
          _stream(stream))


OES_ALIGN_NOALLOC_SCRATCH_BYTES = 1 << 20


def moe_align_block_size_noalloc(ids, R, E, B, ignore_invalid, sorted_ids, block_expert,
                                 n_post_pad, status, stream=None):
    _call("moe_align_block_size_noalloc", _ptr(ids), R, E, B, int(bool(ignore_invalid)),
          _ptr(sorted_ids), _ptr(block_expert), _ptr(n_post_pad), _ptr(status), _stream(stream))


# -------------------------------------------------------------------- GEMM
def oes_tile_plan(R, E) -> int:
    b = C.c_int()
    _call("oes_tile_plan", R, E, C.byref(b))
    return b.value


def routed_experts(layer, E, e2s, wfmt, pool, row_bytes, S, H, I, input_scale13=None,
                   input_scale2=None) -> RoutedExperts:
    return RoutedExperts(layer, E, _ptr(e2s), wfmt, _ptr(pool), row_bytes, S, H, I,
                         _ptr(input_scale13), _ptr(input_scale2))


def moe_grouped_gemm_workspace_size(view: RoutedExperts, T, k) -> int:
    return int(load().moe_grouped_gemm_workspace_size(C.byref(view), T, k))


def moe_grouped_gemm_slots(view: RoutedExperts, x, T, k, ids, weights, sorted_ids, block_expert,
                           n_post_pad, B, workspace, workspace_bytes, out, status, stream=None):
    _call("moe_grouped_gemm_slots", C.byref(view), _ptr(x), T, k, _ptr(ids), _ptr(weights),
          _ptr(sorted_ids), _ptr(block_expert), _ptr(n_post_pad), B, _ptr(workspace),
          workspace_bytes, _ptr(out), _ptr(status), _stream(stream))


# ------------------------------------------------------------- whole layer
def layer_desc(E, H, I, wfmt, input_scale13=None, input_scale2=None) -> LayerDesc:
    return LayerDesc(E, H, I, wfmt, _ptr(input_scale13), _ptr(input_scale2))


def chunk(x, T, k, out, status, workspace, workspace_bytes, logits=None, gate=None) -> Chunk:
    return Chunk(_ptr(logits), _ptr(gate), _ptr(x), T, k, _ptr(out), _ptr(status), _ptr(workspace),
                 workspace_bytes)


def moe_layer_workspace_size(desc: LayerDesc, T, k) -> int:
    return int(load().moe_layer_workspace_size(C.byref(desc), T, k))


def moe_layer_workspace_views(desc: LayerDesc, T, k, workspace) -> dict:
    ps = [C.c_void_p() for _ in range(7)]
    _call("moe_layer_workspace_views", C.byref(desc), T, k, _ptr(workspace), *[C.byref(p) for p in ps])
    names = ["ids", "weights", "distinct", "d_count", "sorted_ids", "block_expert", "n_post_pad"]
    return {n: p.value for n, p in zip(names, ps)}


def moe_layer_forward_slots(cache, src, pool, layer, desc: LayerDesc, ch: Chunk, record_stats,
                            stream=None):
    _call("moe_layer_forward_slots", cache, src, _ptr(pool), layer, C.byref(desc), C.byref(ch),
          int(bool(record_stats)), _stream(stream))


def moe_layer_forward_stream(src, layer_buf, layer, desc: LayerDesc, ch: Chunk, copy_stream=None,
                             compute_stream=None):
    _call("moe_layer_forward_stream", src, _ptr(layer_buf), layer, C.byref(desc), C.byref(ch),
          _stream(copy_stream), _stream(compute_stream))


def oes_takes_slot_path(T, k, E, S, demand_tokens) -> bool:
    return bool(load().oes_takes_slot_path(T, k, E, S, demand_tokens))


def moe_layer_forward(cache, src, pool, layer_buf, layer, desc: LayerDesc, ch: Chunk, demand_tokens,
                      record_stats, copy_stream=None, stream=None) -> bool:
    """Returns True when the chunk took the slot path."""
    took = C.c_int(-1)
    _call("moe_layer_forward", cache, src, _ptr(pool), _ptr(layer_buf), layer, C.byref(desc),
          C.byref(ch), demand_tokens, int(bool(record_stats)), _stream(copy_stream), _stream(stream),
          C.byref(took))
    return bool(took.value)


def oes_stage_plan_create(cache, layers, skip_resident, stream=None):
    arr = (_i * len(layers))(*[int(l) for l in layers])
    out = _vp()
    _call("oes_stage_plan_create", cache, arr, len(layers), int(bool(skip_resident)),
          _stream(stream), C.byref(out))
    return out.value


def oes_stage_plan_destroy(plan):
    _call("oes_stage_plan_destroy", plan)


def oes_stage_plan_layer(plan, i, E):
    """(runs as a list of (e0, e1), staged rows) of layer i of the plan."""
    n, rows = _i(), _i()
    buf = (C.c_int32 * (2 * E))()
    _call("oes_stage_plan_layer", plan, i, C.byref(n), C.cast(buf, _vp), C.byref(rows))
    return [(buf[2 * j], buf[2 * j + 1]) for j in range(n.value)], rows.value


def moe_layers_forward_staged(plan, src, pool, desc: LayerDesc, chunks, copy_stream=None,
                              compute_stream=None):
    arr = (Chunk * len(chunks))(*chunks)
    _call("moe_layers_forward_staged", plan, src, _ptr(pool), C.byref(desc), arr,
          _stream(copy_stream), _stream(compute_stream))


def moe_grouped_gemm_workspace_views(view, T, k, workspace) -> dict:
    ps = [C.c_void_p() for _ in range(3)]
    _call("moe_grouped_gemm_workspace_views", C.byref(view), T, k, _ptr(workspace),
          *[C.byref(p) for p in ps])
    return {n: p.value for n, p in zip(["h", "y", "x16"], ps)}


def slot_cache_ensure_tagged(cache, layer, experts, n, record_stats, tag, miss, n_miss, status,
                             stream=None):
    _call("slot_cache_ensure_tagged", cache, layer, _ptr(experts), n, int(bool(record_stats)), tag,
          _ptr(miss), _ptr(n_miss), _ptr(status), _stream(stream))


def slot_cache_set_policy(cache, policy, lrfu_k=0):
    _call("slot_cache_set_policy", cache, policy, lrfu_k)


def slot_cache_read_lrfu(cache, S, stream=None):
    crf = np.zeros(S, np.uint64)
    pin = np.zeros(S, np.int32)
    _call("slot_cache_read_lrfu", cache, crf.ctypes.data, pin.ctypes.data, _stream(stream))
    return crf, pin
