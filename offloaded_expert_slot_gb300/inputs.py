"""Seeded synthetic inputs for the offloaded-MoE slot path.

This module only PRODUCES data: router inputs, expert weights in the host
source's byte layout, the pre-filled state of a slot pool, and routed ids for
the standalone align sweep.  It holds none of the path's arithmetic (no
routing, no LRU, no alignment, no expert MLP, no NVFP4 decoding), so the CUDA
path and the CPU oracle can both consume what it makes without sharing code.

Random numbers: numpy PCG64 for everything small (router inputs, pool state,
routed ids), which is identical on every platform; torch's generator for the
bulk expert weights, on the device the caller names (CUDA when gigabytes are
needed).  The bytes it returns are the ground truth both sides read.

Encodings produced here (data formats, not path arithmetic):
  * bf16 is IEEE binary32 rounded to nearest-even in its top 16 bits.
  * NVFP4 weights: per expert and per matrix a global fp32 scale
    gs = amax / (6 * 448); per 16 consecutive K elements an e4m3 scale
    sc = e4m3(amax16 / (6 * gs)) (round to nearest even, at most 448); each
    value q = e2m1(w / (sc * gs)) rounded to nearest with ties to even on
    the grid {0, 0.5, 1, 1.5, 2, 3, 4, 6} and saturated at 6.  An all-zero
    block gets sc = 0 and q = 0.  This is the plainest reading of "e2m1
    values, e4m3 per-16 block scales, fp32 per-tensor scale".
"""
from __future__ import annotations

import math

import numpy as np
import torch

from .configs import LayerConfig, expert_row_bytes, nvfp4_offsets

WEIGHT_STD = 0.02


# ---------------------------------------------------------------- helpers
def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_torch(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


# ---------------------------------------------------------------- router inputs
def router_inputs(cfg: LayerConfig) -> dict:
    """x [T, H] as bf16 bits; logits [T, E] fp32, or the gate [H, E] as bf16 bits.

    x ~ N(0, 1).  Router logits ~ N(0, 1) fp32; with "normal+zipf" every
    expert e also gets the bias -s * ln(rank[e]) for a seeded permutation
    rank of 1..E, so the router prefers a Zipf(s) set of hot experts.  With
    "gate" the logits are not given: a bf16 gate [H, E] ~ N(0, 0.02) is.
    """
    g = rng(cfg.seed)
    out = {}
    out["x"] = f32_to_bf16_bits(g.standard_normal((cfg.T, cfg.H), dtype=np.float32))
    if cfg.logits == "gate":
        out["gate"] = f32_to_bf16_bits(
            (g.standard_normal((cfg.H, cfg.E), dtype=np.float32) * WEIGHT_STD))
        out["logits"] = None
    else:
        logits = g.standard_normal((cfg.T, cfg.E), dtype=np.float32)
        if cfg.logits == "normal+zipf":
            rank = g.permutation(cfg.E) + 1
            bias = (-cfg.zipf_s * np.log(rank.astype(np.float64))).astype(np.float32)
            logits = (logits + bias[None, :]).astype(np.float32)
        out["logits"] = np.ascontiguousarray(logits)
        out["gate"] = None
    return out


# ---------------------------------------------------------------- pool state
def pool_prefill(cfg: LayerConfig) -> dict:
    """Seeded pre-filled pool: `prefill` distinct (layer, expert) keys at seeded
    slots with a seeded, strictly ordered recency (timestamps 1..prefill).

    key = layer * E + expert.  Empty slots hold key -1 and timestamp 0.
    clock = the last timestamp handed out.
    """
    g = rng(cfg.seed + 7919)
    S, n = cfg.S, cfg.prefill
    slot_key = np.full(S, -1, dtype=np.int32)
    slot_ts = np.zeros(S, dtype=np.int64)
    if n:
        keys = g.choice(cfg.L * cfg.E, size=n, replace=False).astype(np.int32)
        slots = g.permutation(S)[:n]
        ts = g.permutation(n).astype(np.int64) + 1
        slot_key[slots] = keys
        slot_ts[slots] = ts
    return {"slot_key": slot_key, "slot_ts": slot_ts, "clock": int(n)}


# ---------------------------------------------------------------- align sweep ids
def uniform_routes(T: int, k: int, E: int, seed: int) -> np.ndarray:
    """T tokens each routed to k distinct experts drawn uniformly, flattened [T*k] int32."""
    g = rng(seed)
    out = np.empty((T, k), dtype=np.int32)
    step = max(1, (1 << 22) // max(E, 1))
    for t0 in range(0, T, step):
        t1 = min(T, t0 + step)
        u = g.random((t1 - t0, E), dtype=np.float32)
        out[t0:t1] = np.argpartition(u, k - 1, axis=1)[:, :k]
    return out.reshape(-1)


# ---------------------------------------------------------------- NVFP4 encoder
def _e2m1_codes(v: torch.Tensor) -> torch.Tensor:
    """Round to nearest e2m1 (ties to even mantissa), saturate at 6; 4-bit codes."""
    m = v.abs()
    idx = ((m > 0.25).to(torch.uint8) + (m >= 0.75).to(torch.uint8) + (m > 1.25).to(torch.uint8)
           + (m >= 1.75).to(torch.uint8) + (m > 2.5).to(torch.uint8) + (m >= 3.5).to(torch.uint8)
           + (m > 5.0).to(torch.uint8))
    neg = (v < 0) & (idx > 0)
    return idx | (neg.to(torch.uint8) << 3)


def quantize_nvfp4(w: torch.Tensor):
    """Encode w [n, rows, K] fp32 (n experts of one matrix) as NVFP4.

    Returns (values [n, rows, K/2] u8, scales [n, K/64, rows, 4] u8 e4m3,
    global scales [n] fp32).
    """
    n, rows, K = w.shape
    assert K % 64 == 0
    amax = w.abs().amax(dim=(1, 2))
    gs = amax / (6.0 * 448.0)
    gs = torch.where(gs > 0, gs, torch.ones_like(gs))
    blk = w.reshape(n, rows, K // 16, 16)
    amax16 = blk.abs().amax(dim=-1)
    sc8 = (amax16 / (6.0 * gs[:, None, None])).clamp(max=448.0).to(torch.float8_e4m3fn)
    denom = sc8.to(torch.float32) * gs[:, None, None]
    safe = torch.where(denom > 0, denom, torch.ones_like(denom))
    v = torch.where(denom[..., None] > 0, blk / safe[..., None], torch.zeros_like(blk))
    codes = _e2m1_codes(v).reshape(n, rows, K)
    packed = codes[..., 0::2] | (codes[..., 1::2] << 4)
    sc_bytes = sc8.view(torch.uint8).reshape(n, rows, K // 64, 4).permute(0, 2, 1, 3).contiguous()
    return packed.contiguous(), sc_bytes, gs.to(torch.float32)


# ---------------------------------------------------------------- expert source
def _expert_generator(cfg: LayerConfig, layer: int, e: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(((cfg.seed * 1_000_003 + 17 * layer) * 65_537 + e) & ((1 << 62) - 1))
    return g


def expert_rows(cfg: LayerConfig, layer: int, experts, device="cpu") -> torch.Tensor:
    """Rows of the given experts of one layer in the host-source byte layout,
    [len(experts), row_bytes] u8 on `device`.  Every expert has its own
    seeded generator, so any subset can be regenerated on its own.

    Weights ~ N(0, 0.02) drawn as fp32 and rounded to bf16; NVFP4 rows encode
    those bf16 values (see module docstring).
    """
    E, H, I = cfg.E, cfg.H, cfg.I
    rb = expert_row_bytes(cfg.wfmt, H, I)
    experts = list(experts)
    n = len(experts)
    w13 = torch.empty((n, 2 * I, H), dtype=torch.bfloat16, device=device)
    w2 = torch.empty((n, H, I), dtype=torch.bfloat16, device=device)
    for i, e in enumerate(experts):
        g = _expert_generator(cfg, layer, int(e), device)
        w13[i] = (torch.randn((2 * I, H), generator=g, device=device) * WEIGHT_STD).to(torch.bfloat16)
        w2[i] = (torch.randn((H, I), generator=g, device=device) * WEIGHT_STD).to(torch.bfloat16)
    rows = torch.empty((n, rb), dtype=torch.uint8, device=device)
    if cfg.wfmt == "bf16":
        rows[:, : 2 * I * H * 2] = w13.reshape(n, -1).view(torch.uint8)
        rows[:, 2 * I * H * 2:] = w2.reshape(n, -1).view(torch.uint8)
    else:
        scale_in = 0.0
        if cfg.layer_input_scales:
            scale_in = float(cfg.layer_input_scales[layer % len(cfg.layer_input_scales)])
        o = nvfp4_offsets(H, I)
        q13, s13, gs13 = quantize_nvfp4(w13.to(torch.float32))
        q2, s2, gs2 = quantize_nvfp4(w2.to(torch.float32))
        rows[:, o["w13q"]:o["w13s"]] = q13.reshape(n, -1)
        rows[:, o["w13s"]:o["w2q"]] = s13.reshape(n, -1)
        rows[:, o["w2q"]:o["w2s"]] = q2.reshape(n, -1)
        rows[:, o["w2s"]:o["scalars"]] = s2.reshape(n, -1)
        scal = torch.stack([gs13, gs2, torch.full_like(gs13, scale_in),
                            torch.full_like(gs13, scale_in)], dim=1).contiguous()
        rows[:, o["scalars"]:o["end"]] = scal.view(torch.uint8).reshape(n, 16)
    return rows


def expert_layer_rows(cfg: LayerConfig, layer: int, device="cpu", out: torch.Tensor | None = None,
                      chunk: int = 32) -> torch.Tensor:
    """All E expert rows of one layer, [E, row_bytes] u8, generated on
    `device` (in chunks) and written into `out` (any device, e.g. pinned host
    memory) when given.  Row e equals expert_rows(cfg, layer, [e]) made on
    the same kind of device."""
    rb = expert_row_bytes(cfg.wfmt, cfg.H, cfg.I)
    if out is None:
        out = torch.empty((cfg.E, rb), dtype=torch.uint8)
    for e0 in range(0, cfg.E, chunk):
        e1 = min(cfg.E, e0 + chunk)
        out[e0:e1].copy_(expert_rows(cfg, layer, range(e0, e1), device=device))
    return out


def empty_slot_row(cfg: LayerConfig) -> np.ndarray:
    """Content of a slot that holds no expert: zeros, and for NVFP4 the
    'other slots' input scale in both input-scale fields."""
    row = np.zeros(cfg.row_bytes, dtype=np.uint8)
    if cfg.wfmt == "nvfp4" and cfg.other_slot_input_scale:
        o = nvfp4_offsets(cfg.H, cfg.I)
        sc = np.array([0.0, 0.0, cfg.other_slot_input_scale, cfg.other_slot_input_scale],
                      dtype=np.float32)
        row[o["scalars"]:o["end"]] = sc.view(np.uint8)
    return row


def source_layer_index(cfg: LayerConfig, layer: int) -> int:
    """Which distinct pinned source buffer backs `layer` (all distinct unless the
    config caps the number of distinct source layers to bound host memory)."""
    if cfg.distinct_source_layers:
        return layer % cfg.distinct_source_layers
    return layer


def n_source_buffers(cfg: LayerConfig) -> int:
    return cfg.distinct_source_layers or cfg.L


def gib(nbytes: int) -> float:
    return nbytes / float(1 << 30)


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("annotations", "math")]
