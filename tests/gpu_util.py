"""Helpers shared by the GPU tests: device buffers and workload set-up.

Only data plumbing lives here (allocation, copies, seeded inputs from the
generator module); every step of the path under test runs in liboes.
"""
from __future__ import annotations

import numpy as np
import torch

from offloaded_expert_slot_gb300 import build, oes
from offloaded_expert_slot_gb300.configs import LayerConfig
from offloaded_expert_slot_gb300.inputs import (empty_slot_row, expert_layer_rows, n_source_buffers,
                                                pool_prefill, router_inputs, source_layer_index)

_built = False


def lib():
    global _built
    if not _built:
        build.build()
        _built = True
    return oes.load()


def cuda(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def i32(n, fill=0) -> torch.Tensor:
    return torch.full((max(int(n), 1),), fill, dtype=torch.int32, device="cuda")


def f32(n) -> torch.Tensor:
    return torch.zeros(max(int(n), 1), dtype=torch.float32, device="cuda")


def scratch(nbytes: int) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device="cuda")


def bits16(bits: np.ndarray) -> torch.Tensor:
    """uint16 bit patterns -> CUDA int16 tensor with the same bits."""
    return cuda(np.ascontiguousarray(bits).view(np.int16))


def status() -> torch.Tensor:
    return i32(1, 0)


class Workload:
    """One layer config set up on the GPU: router inputs, pinned host source,
    slot pool with the seeded pre-fill, slot cache and expert source handles."""

    def __init__(self, cfg: LayerConfig, with_pool: bool = True, gen_device: str = "cuda",
                 extra_rows: int = 0):
        lib()
        self.cfg = cfg
        self.rin = router_inputs(cfg)
        self.x = bits16(self.rin["x"])
        self.logits = cuda(self.rin["logits"]) if self.rin["logits"] is not None else None
        self.gate = bits16(self.rin["gate"]) if self.rin["gate"] is not None else None
        rb = cfg.row_bytes
        nsrc = n_source_buffers(cfg)
        self.src_bufs = []
        for l in range(nsrc):
            buf = torch.empty((cfg.E, rb), dtype=torch.uint8, pin_memory=True)
            expert_layer_rows(cfg, l, device=gen_device, out=buf)
            self.src_bufs.append(buf)
        self.src_np = [b.numpy() for b in self.src_bufs]
        bases = [self.src_bufs[source_layer_index(cfg, l)] for l in range(cfg.L)]
        self.src = oes.oes_expert_source_create(bases, cfg.E, rb)
        self.cache = None
        self.pool = None
        if with_pool:
            # rows past S (the staging buffers of the staged runner) start as
            # a byte pattern no expert row has
            self.pool_all = torch.full((cfg.S + extra_rows, rb), 0x5A, dtype=torch.uint8,
                                       device="cuda")
            self.pool = self.pool_all[:cfg.S]
            self.cache = oes.slot_cache_create(cfg.S, cfg.L, cfg.E)
            self.reset_pool()

    def source_row(self, layer: int, e: int) -> np.ndarray:
        return self.src_np[source_layer_index(self.cfg, layer)][e]

    def reset_pool(self):
        """Seeded pre-fill: tables and the bytes of every pre-filled slot."""
        cfg = self.cfg
        st = pool_prefill(cfg)
        self.prefill = st
        oes.slot_cache_load_state(self.cache, st["slot_key"], st["slot_ts"], st["clock"])
        empty = torch.from_numpy(empty_slot_row(cfg)).cuda()
        self.pool[:] = empty
        for s in np.nonzero(st["slot_key"] >= 0)[0]:
            k = int(st["slot_key"][s])
            self.pool[int(s)].copy_(torch.from_numpy(self.source_row(k // cfg.E, k % cfg.E)))
        torch.cuda.synchronize()

    def oracle_pool(self) -> dict:
        """The oracle's model of the pre-filled pool: slot -> row bytes."""
        cfg = self.cfg
        empty = empty_slot_row(cfg)
        return {s: (self.source_row(int(k) // cfg.E, int(k) % cfg.E) if k >= 0 else empty)
                for s, k in enumerate(self.prefill["slot_key"])}

    def close(self):
        if self.cache:
            oes.slot_cache_destroy(self.cache)
            self.cache = None
        if self.src:
            oes.oes_expert_source_destroy(self.src)
            self.src = None


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()
