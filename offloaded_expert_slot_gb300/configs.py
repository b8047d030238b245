"""The five workloads of the offloaded-MoE slot path, by name and size.

Each workload is shaped like the ones on the source pages (FreeToken PR #676
"--moe-prefill-demand-tokens", sections Problem, Tests and A/B; gdevenyi's
review comment on the same page; vLLM fork PR #48, section What): 512 experts
at top-10 with hidden 2048 and expert intermediate 768, 1100- or 1650-slot
pools shared by several layers, and chunks from decode width (32 tokens) to
4096 tokens.  The first workload is a tiny one that a plain CPU model of the
path finishes in milliseconds.

Nothing here computes any step of the path; it only names sizes.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace


@dataclass(frozen=True)
class LayerConfig:
    name: str
    T: int                 # tokens in the chunk
    k: int                 # top-k
    E: int                 # the layer's expert count
    H: int                 # hidden size
    I: int                 # expert intermediate size
    wfmt: str              # "bf16" or "nvfp4"
    S: int                 # slots in the pool
    L: int                 # layers whose experts share the pool
    prefill: int           # slots pre-filled with seeded (layer, expert) pairs
    query_width: int       # ids per LRU ensure query
    logits: str            # "gate" | "normal" | "normal+zipf"
    zipf_s: float = 0.0    # Zipf exponent of the per-expert logit bias
    layer: int = 0         # layer that is forwarded
    seed: int = 0
    # NVFP4 only: the forwarded layers' input scales and the value every
    # other slot carries (FreeToken PR #676, Tests: the layer's scales are
    # 2.0 and 3.0, every slot holds 9.0).
    layer_input_scales: tuple = ()
    other_slot_input_scale: float = 0.0
    distinct_source_layers: int = 0   # 0: one pinned source per layer
    # NVFP4 only: activations quantised to NVFP4 too (W4A4), under the
    # maximum of the layer's input scales
    w4a4: bool = False

    @property
    def R(self) -> int:
        return self.T * self.k

    @property
    def row_bytes(self) -> int:
        return expert_row_bytes(self.wfmt, self.H, self.I)


def expert_row_bytes(wfmt: str, H: int, I: int) -> int:
    """Bytes of one expert row in the host source and in a pool slot.

    bf16 row: w13 [2I, H] bf16, then w2 [H, I] bf16.
    nvfp4 row: w13 values [2I, H/2] u8 (two e2m1 per byte, element 2i in the
    low nibble), w13 scales [H/64, 2I, 4] e4m3 (K-chunk-major: the four
    16-element scales of a 64-wide K chunk of one row are one 32-bit word),
    w2 values [H, I/2] u8, w2 scales [I/64, H, 4] e4m3, then four fp32
    scalars: global scale of w13, global scale of w2, input scale of w13,
    input scale of w2.  Every section starts on a 16-byte boundary.
    """
    if wfmt == "bf16":
        return 2 * I * H * 2 + H * I * 2
    if wfmt == "nvfp4":
        assert H % 64 == 0 and I % 64 == 0
        return (2 * I * H // 2) + (2 * I * H // 16) + (H * I // 2) + (H * I // 16) + 16
    raise ValueError(wfmt)


def nvfp4_offsets(H: int, I: int) -> dict:
    """Byte offsets of the sections of an NVFP4 expert row (see expert_row_bytes)."""
    o = {}
    o["w13q"] = 0
    o["w13s"] = o["w13q"] + 2 * I * H // 2
    o["w2q"] = o["w13s"] + 2 * I * H // 16
    o["w2s"] = o["w2q"] + H * I // 2
    o["scalars"] = o["w2s"] + H * I // 16
    o["end"] = o["scalars"] + 16
    return o


C1 = LayerConfig(name="c1_tiny", T=16, k=2, E=8, H=128, I=64, wfmt="bf16", S=6, L=1,
                 prefill=3, query_width=4, logits="gate", seed=1001)
C2 = LayerConfig(name="c2_decode_width", T=32, k=10, E=512, H=2048, I=768, wfmt="bf16",
                 S=1100, L=2, prefill=800, query_width=128, logits="normal", seed=1002)
C3 = LayerConfig(name="c3_short_prefill", T=200, k=10, E=512, H=2048, I=768, wfmt="bf16",
                 S=1100, L=2, prefill=800, query_width=128, logits="normal+zipf", zipf_s=1.1,
                 seed=1003)
C4 = LayerConfig(name="c4_nvfp4_prefill", T=600, k=10, E=512, H=2048, I=768, wfmt="nvfp4",
                 S=1100, L=2, prefill=800, query_width=128, logits="normal", seed=1004,
                 layer_input_scales=(2.0, 3.0), other_slot_input_scale=9.0)
C5 = LayerConfig(name="c5_long_prefill", T=4096, k=10, E=512, H=2048, I=768, wfmt="nvfp4",
                 S=1650, L=48, prefill=0, query_width=128, logits="normal", seed=1005)

CONFIGS = {c.name: c for c in (C1, C2, C3, C4, C5)}


@dataclass(frozen=True)
class AlignSweep:
    """Standalone moe_align_block_size sweep: tokens x top-k uniformly routed."""
    T: int = 8192
    k: int = 8
    Es: tuple = (1023, 2100)
    block: int = 64
    seed: int = 1006


C5B = AlignSweep()


def scaled(cfg: LayerConfig, **kw) -> LayerConfig:
    """A copy of cfg with some sizes replaced (small parity cases)."""
    return replace(cfg, **kw)
