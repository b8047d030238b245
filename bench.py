"""Benchmark: routed tokens/s of one offloaded-MoE layer forward over the GPU
slot cache, on one GB300 (or N independent replicas, one per GPU).

A step is one pass of the whole slot path over one chunk: route -> distinct
experts -> queries of 128 (ensure + miss copies from pinned host memory) ->
align -> grouped SwiGLU GEMM -> combine.  Before each step the cache tables
are restored on the device to the workload's seeded state (a device-to-device
copy of the tables inside the timed region), so every step admits the same
misses and copies the same rows.

Headline workload: the long prefill, the largest single-GPU workload -- a
4096-token chunk, top-10 over 512 NVFP4 experts (hidden 2048, intermediate
768), a 1650-slot pool shared by 48 layers that starts empty, so every step
loads all of the layer's routed experts (1.36 GB) over the host link and
runs the GEMM over them.  Only the forwarded layer's rows are pinned on the
host: with an empty pool no other layer's row is ever read.  The
decode-width step (32 tokens, bf16 experts, 1100 slots with 800 pre-filled)
is measured after it and reported under "decode_width".

Output: one JSON line (rank 0).  `value` = tokens of all ranks / max step time
over ranks; `e2e` = the same through the C ABI with the chunk's inputs copied
from pinned host memory and the output read back inside every timed step;
`roofline` = the step with the largest share of the step time, against its
bound; `roofline_gemm` = the grouped GEMM against its own bound (tensor
cores or HBM, whichever is slower for its flops and bytes); `cpu_baseline` =
the CPU oracle timed on the host cores on a bounded sample of the same
workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

# The CPU oracle (cpu_baseline and --impl reference) does its matrix products
# in numpy's BLAS and everything else in single-threaded Python.  The BLAS
# thread pool is sized here, before numpy loads it, to the cores this process
# may run on, and the baselines report that number.
CPU_THREADS = len(os.sched_getaffinity(0))
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(CPU_THREADS))

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from offloaded_expert_slot_gb300.configs import CONFIGS  # noqa: E402

DEFAULT_CONFIG = "c5_long_prefill"
SECONDARY_CONFIG = "c2_decode_width"
METRIC = "routed tokens/s per MoE layer (1xGB300)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of the launches
# the breakdown times, from one ncu capture of the current kernels on each
# workload: per whole-query copy_misses_kernel launch, and per step for the
# grouped GEMM (GEMM1, GEMM2, combine).  A workload without an entry, or a
# kernel changed since its capture, reports traffic null.
TRAFFIC = {
    "c2_decode_width": {"copy_per_launch": 123.77e6, "gemm_per_step": 2342.5e6},
    "c5_long_prefill": {"copy_per_launch": 275.66e6, "gemm_per_step": 1934.1e6},
}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        d["source"] = "measured"
        return d
    d = dict(FALLBACK_PEAKS)
    d["source"] = "fallback"
    return d


# ----------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- oracle
ORACLE_SAMPLE_TOKENS = 1024   # chunk prefix the oracle takes per sample
ORACLE_MLP_TOKENS = 8         # of which the expert MLP and combine run on this many


def oracle_chunk(cfg, rin):
    """The oracle's bounded sample of a chunk: its first ORACLE_SAMPLE_TOKENS
    tokens (same experts, pool, weights and query width)."""
    from offloaded_expert_slot_gb300.configs import scaled
    Ts = min(cfg.T, ORACLE_SAMPLE_TOKENS)
    if Ts == cfg.T:
        return cfg, rin
    r = dict(rin)
    r["x"] = rin["x"][:Ts]
    if rin.get("logits") is not None:
        r["logits"] = rin["logits"][:Ts]
    return scaled(cfg, T=Ts), r


def oracle_sample(cfg, rin, source_row, prefill, n_tokens, seed, toks=None):
    """One bounded sample of the oracle's slot path over `cfg`'s chunk:
    routing, distinct experts, every LRU query and the align for the whole
    chunk; the expert MLP and combine for n_tokens sampled tokens (or the
    given `toks`).  Returns seconds."""
    from oracle.layer import forward_slots
    from oracle.slot_cache import SlotCache
    from offloaded_expert_slot_gb300.inputs import empty_slot_row
    empty = empty_slot_row(cfg)
    pool = {s: (source_row(int(k) // cfg.E, int(k) % cfg.E) if k >= 0 else empty)
            for s, k in enumerate(prefill["slot_key"])}
    cache = SlotCache.from_state(cfg.S, cfg.L, cfg.E, prefill["slot_key"], prefill["slot_ts"],
                                 prefill["clock"])
    if toks is None:
        toks = np.random.default_rng(seed).choice(cfg.T, n_tokens, replace=False)
    per = -(-(cfg.T * cfg.k) // cfg.E)           # the library's tile plan: routes per expert
    block = 16 if per <= 8 else 128
    t0 = time.perf_counter()
    forward_slots(cfg, rin, source_row, cache, pool, block=block, tokens=toks)
    return time.perf_counter() - t0


def sample_text(cfg, cs, n_tok):
    pre = (f"the first {cs.T} of the chunk's {cfg.T} tokens"
           if cs.T < cfg.T else f"the whole {cfg.T}-token chunk")
    return (f"oracle slot path over {pre} (routing, distinct experts, LRU queries, align; "
            f"the workload's experts, pool and weights) with the expert MLP and combine for "
            f"{n_tok} of those tokens; its matrix products on numpy's BLAS with {blas_threads()} "
            f"threads, the rest single-threaded Python")


def lazy_source(cfg, needed):
    """Host rows of the (layer, expert) pairs in `needed`, generated on the CPU."""
    from offloaded_expert_slot_gb300.inputs import expert_rows
    rows = {}
    by_layer = {}
    for l, e in needed:
        by_layer.setdefault(l, []).append(e)
    for l, es in by_layer.items():
        es = sorted(set(es))
        r = expert_rows(cfg, l, es).numpy()
        for i, e in enumerate(es):
            rows[(l, e)] = r[i]
    return lambda l, e: rows[(l, e)]


def reference_arm(args, cfg):
    """The CPU oracle as the reference implementation, on the host cores.
    The MLP sample is one fixed set of tokens, so that only their experts'
    rows need generating on the host (about 0.2 s an NVFP4 expert); every
    other expert the chunk loads gets a zero row, which the sample never
    reads."""
    from offloaded_expert_slot_gb300.inputs import pool_prefill, router_inputs
    from oracle.router import gate_logits, route_topk
    cs, rin = oracle_chunk(cfg, router_inputs(cfg))
    prefill = pool_prefill(cfg)
    logits = rin["logits"] if rin["logits"] is not None else gate_logits(rin["x"], rin["gate"])
    ids, _ = route_topk(logits, cfg.k)
    n_tok = min(cs.T, ORACLE_MLP_TOKENS)
    toks = np.random.default_rng(cfg.seed).choice(cs.T, n_tok, replace=False)
    needed = {(cfg.layer, int(e)) for e in np.unique(ids[toks])}
    src = lazy_source(cfg, needed)
    zero = np.zeros(cfg.row_bytes, np.uint8)
    src_row = lambda l, e: src(l, e) if (l, e) in needed else zero
    for i in range(args.warmup):
        oracle_sample(cs, rin, src_row, prefill, n_tok, i, toks=toks)
    times = [oracle_sample(cs, rin, src_row, prefill, n_tok, 100 + i, toks=toks)
             for i in range(args.steps)]
    s = float(np.sum(times))
    value = n_tok * args.steps / s
    cores = blas_threads()
    sample = sample_text(cfg, cs, n_tok) + " (a fixed token sample, the same every step)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000 * s / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(cfg, args.gpus),
            "cpu_baseline": {"kind": "oracle", "value": value, "unit": "tokens/s", "cores": cores,
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ----------------------------------------------------------------- GPU arm
class Bench:
    def __init__(self, cfg, rank):
        import torch

        from offloaded_expert_slot_gb300 import oes
        from offloaded_expert_slot_gb300.inputs import (empty_slot_row, expert_layer_rows,
                                                        n_source_buffers, pool_prefill,
                                                        router_inputs, source_layer_index)
        from offloaded_expert_slot_gb300.configs import scaled
        if cfg.prefill == 0 and cfg.layer == 0 and not cfg.distinct_source_layers:
            # an empty pool only ever reads the forwarded layer's rows: pin
            # that layer alone and let every layer's source point at it
            cfg = scaled(cfg, distinct_source_layers=1)
        self.torch, self.oes, self.cfg = torch, oes, cfg
        oes.load()
        rb = cfg.row_bytes
        self.rin = router_inputs(cfg)
        self.src_bufs = []
        for l in range(n_source_buffers(cfg)):
            buf = torch.empty((cfg.E, rb), dtype=torch.uint8, pin_memory=True)
            expert_layer_rows(cfg, l, device="cuda", out=buf)
            self.src_bufs.append(buf)
        self.source_index = lambda l: source_layer_index(cfg, l)
        bases = [self.src_bufs[source_layer_index(cfg, l)] for l in range(cfg.L)]
        self.src = oes.oes_expert_source_create(bases, cfg.E, rb)
        self.pool = torch.empty((cfg.S, rb), dtype=torch.uint8, device="cuda")
        self.cache = oes.slot_cache_create(cfg.S, cfg.L, cfg.E)
        st = pool_prefill(cfg)
        self.prefill = st
        oes.slot_cache_load_state(self.cache, st["slot_key"], st["slot_ts"], st["clock"])
        self.pool[:] = torch.from_numpy(empty_slot_row(cfg)).cuda()
        for s in np.nonzero(st["slot_key"] >= 0)[0]:
            k = int(st["slot_key"][s])
            self.pool[int(s)].copy_(self.src_bufs[source_layer_index(cfg, k // cfg.E)][k % cfg.E])
        self.snap = torch.empty(oes.slot_cache_state_bytes(self.cache), dtype=torch.uint8,
                                device="cuda")
        oes.slot_cache_snapshot(self.cache, self.snap)
        self.x = torch.from_numpy(self.rin["x"].view(np.int16)).cuda()
        self.logits = torch.from_numpy(self.rin["logits"]).cuda()
        self.wfmt = oes.OES_WFMT_BF16 if cfg.wfmt == "bf16" else oes.OES_WFMT_NVFP4
        self.desc = oes.layer_desc(cfg.E, cfg.H, cfg.I, self.wfmt)
        self.wsb = oes.moe_layer_workspace_size(self.desc, cfg.T, cfg.k)
        self.ws = torch.empty(self.wsb, dtype=torch.uint8, device="cuda")
        self.out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.chunk = oes.chunk(self.x, cfg.T, cfg.k, self.out, self.status, self.ws, self.wsb,
                               logits=self.logits)
        torch.cuda.synchronize()

    def step(self):
        oes = self.oes
        oes.slot_cache_restore(self.cache, self.snap)
        oes.moe_layer_forward_slots(self.cache, self.src, self.pool, self.cfg.layer, self.desc,
                                    self.chunk, 0)

    def timed(self, fn, steps):
        torch = self.torch
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    # -- the same step as one CUDA graph, replayed
    def graph_timed(self, steps, warmup):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                self.step()
        torch.cuda.current_stream().wait_stream(s)
        for _ in range(warmup):
            g.replay()
        ms = self.timed(g.replay, steps)
        st = int(self.status.item())
        if st:
            raise RuntimeError(f"device status {st} after graph replays")
        del g
        return ms

    # -- end to end through the C ABI with host buffers
    def e2e(self, steps, warmup):
        torch, oes, cfg = self.torch, self.oes, self.cfg
        xh = torch.from_numpy(self.rin["x"].view(np.int16)).pin_memory()
        lh = torch.from_numpy(self.rin["logits"]).pin_memory()
        oh = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory()

        def one():
            self.x.copy_(xh, non_blocking=True)
            self.logits.copy_(lh, non_blocking=True)
            self.step()
            oh.copy_(self.out, non_blocking=True)

        for _ in range(warmup):
            one()
        ms = self.timed(one, steps)
        bi = xh.numel() * 2 + lh.numel() * 4
        bo = oh.numel() * 2
        return ms, bi, bo

    # -- per-step breakdown: the same calls, one by one, with events between
    def breakdown(self, steps):
        torch, oes, cfg = self.torch, self.oes, self.cfg
        T, k, E = cfg.T, cfg.k, cfg.E
        R = T * k
        B = oes.oes_tile_plan(R, E)
        cap = oes.align_capacity(R, E, B)
        ids = torch.empty(R, dtype=torch.int32, device="cuda")
        w = torch.empty(R, dtype=torch.float32, device="cuda")
        Lq = min(R, E)
        dist = torch.empty(Lq, dtype=torch.int32, device="cuda")
        dcnt = torch.empty(1, dtype=torch.int32, device="cuda")
        miss = torch.empty(3 * 128, dtype=torch.int32, device="cuda")
        nmiss = torch.empty(1, dtype=torch.int32, device="cuda")
        nmiss_tot = torch.zeros(1, dtype=torch.int32, device="cuda")
        srt = torch.empty(cap, dtype=torch.int32, device="cuda")
        bexp = torch.empty(cap // B, dtype=torch.int32, device="cuda")
        npp = torch.empty(1, dtype=torch.int32, device="cuda")
        awsb = oes.moe_align_workspace_size(R, E, B)
        aws = torch.empty(max(awsb, 256), dtype=torch.uint8, device="cuda")
        e2s = oes.slot_cache_layer_map(self.cache, cfg.layer)
        view = oes.routed_experts(cfg.layer, E, e2s, self.wfmt, self.pool, cfg.row_bytes, cfg.S,
                                  cfg.H, cfg.I)
        gwsb = oes.moe_grouped_gemm_workspace_size(view, T, k)
        gws = torch.empty(gwsb, dtype=torch.uint8, device="cuda")
        names = ["restore", "route", "distinct", "ensure", "copy", "align", "gemm"]
        tot = {n: 0.0 for n in names}
        Q = (Lq + 127) // 128
        for it in range(steps + 1):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3 + 2 * Q + 3)]
            i = 0
            ev[i].record(); i += 1
            oes.slot_cache_restore(self.cache, self.snap)
            ev[i].record(); i += 1
            oes.moe_route_topk(self.logits, T, E, k, ids, w)
            ev[i].record(); i += 1
            oes.moe_distinct_experts(ids, R, E, dist, dcnt)
            marks = []
            for q in range(Q):
                n = min(128, Lq - q * 128)
                ev[i].record(); i += 1
                oes.slot_cache_ensure(self.cache, cfg.layer, dist.data_ptr() + 4 * q * 128, n, 0,
                                      miss, nmiss, self.status)
                if it == 0:
                    nmiss_tot.add_(nmiss)
                ev[i].record(); i += 1
                oes.slot_cache_copy_misses(self.src, self.pool, cfg.S, miss, nmiss, n, self.status)
                marks.append(i)
            ev[i].record(); i += 1
            oes.moe_align_block_size(ids, R, E, B, 1, srt, bexp, npp, self.status, aws, awsb)
            ev[i].record(); i += 1
            oes.moe_grouped_gemm_slots(view, self.x, T, k, ids, w, srt, bexp, npp, B, gws, gwsb,
                                       self.out, self.status)
            ev[i].record(); i += 1
            torch.cuda.synchronize()
            if it == 0:
                continue     # warm-up pass (also counts the misses)
            el = [ev[j].elapsed_time(ev[j + 1]) for j in range(i - 1)]
            tot["restore"] += el[0]
            tot["route"] += el[1]
            tot["distinct"] += el[2]
            for q in range(Q):
                tot["ensure"] += el[3 + 2 * q]
                tot["copy"] += el[4 + 2 * q]
            tot["align"] += el[3 + 2 * Q]
            tot["gemm"] += el[4 + 2 * Q]
        ms = {n: v / steps for n, v in tot.items()}
        n_miss = int(nmiss_tot.item())
        n_blocks = int(npp.item()) // B
        D = int(dcnt.item())
        return ms, {"misses": n_miss, "distinct": D, "blocks": n_blocks, "queries": Q, "block": B,
                    "status": int(self.status.item())}

    def link_probe(self):
        torch = self.torch
        n = 1 << 30
        h = torch.empty(n, dtype=torch.uint8, pin_memory=True)
        d = torch.empty(n, dtype=torch.uint8, device="cuda")
        for _ in range(2):
            d.copy_(h, non_blocking=True)
        ms = self.timed(lambda: d.copy_(h, non_blocking=True), 4)
        del h, d
        return n / (ms / 1e3) / 1e9

    def close(self):
        self.oes.slot_cache_destroy(self.cache)
        self.oes.oes_expert_source_destroy(self.src)


def reduce_max(x: float, dist, device) -> float:
    """Max of a per-rank number over all ranks (the slowest rank sets the
    step time of the job); identity on a single process."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_config(cfg, rank: int):
    """The workload of one replica: the same sizes, with rank r > 0 drawing
    its own seeded chunk, pool pre-fill and expert rows (seed + 101 r).
    Replicas share nothing: each has its own cache, pool and source."""
    if rank == 0:
        return cfg
    from offloaded_expert_slot_gb300.configs import scaled
    return scaled(cfg, seed=cfg.seed + 101 * rank)


def job_value(tokens_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job throughput: tokens of all ranks over the slowest rank's step."""
    return tokens_per_rank * world / (ms_max / 1e3)


def gpu_launches(cfg, with_restore=True):
    """Kernels of liboes launched per step of the slot path."""
    R = cfg.T * cfg.k
    Q = (min(R, cfg.E) + 127) // 128
    Lq = min(R, cfg.E)
    align = 1 if R <= 1024 else 3       # one CTA up to 1024 routes, else count/scan/scatter
    # a query of more than 32 ids copies its misses in two parts
    parts = sum(2 if min(128, Lq - 128 * q) > 32 else 1 for q in range(Q))
    # topk, distinct, Q ensures, a copy per part, group flags, align,
    # gemm1/2 over the hits, gemm1/2 per part over its copied experts, combine
    n = 1 + 1 + Q + parts + 1 + align + 2 + 2 * parts + 1
    if with_restore:
        n += 1                          # the step's restore of the cache tables
    if cfg.logits == "gate":
        n += 1
    if cfg.wfmt == "nvfp4":
        n += 2 if cfg.w4a4 else 1       # W4A4: activation scales and x quantised; else x -> f16
    return n


def config_of(cfg, world):
    """The workload as both arms report it: sizes only, nothing measured."""
    routed_rows = min(cfg.T * cfg.k, cfg.E) * cfg.row_bytes
    return {"workload": cfg.name, "T": cfg.T, "k": cfg.k, "E": cfg.E, "H": cfg.H, "I": cfg.I,
            "wfmt": cfg.wfmt, "slots": cfg.S, "layers_in_pool": cfg.L, "prefilled": cfg.prefill,
            "query_width": cfg.query_width, "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2: a step reads up to min(T*k, E) expert rows, "
                  f"{routed_rows / 1e9:.2f} GB"}


def gemm_roofline(cfg, info, ms, pk, traffic):
    """The grouped GEMM of one step (GEMM1 + GEMM2 + combine) against the
    slower of its two bounds for its algorithmic work: R * 6HI flops on the
    tensor cores (f16 or bf16 MMAs, both at the bf16 rate; the breakdown
    times the GEMM alone, so the burst peak) or D expert rows + x + out bytes
    on HBM."""
    R = cfg.T * cfg.k
    flops = R * 6 * cfg.H * cfg.I
    nbytes = info["distinct"] * cfg.row_bytes + cfg.T * cfg.H * 2 * 2
    hbm, bf16 = float(pk["hbm_gbs"]), float(pk["bf16_tflops"])
    t_tensor, t_hbm = flops / (bf16 * 1e12), nbytes / (hbm * 1e9)
    tflops = flops / (ms / 1e3) / 1e12
    gbs = nbytes / (ms / 1e3) / 1e9
    base = {"kernel": "grouped_gemm (gemm1 + gemm2 + combine)", "peak_source": pk["source"],
            "algorithmic_flops": flops, "algorithmic_bytes": nbytes, "launch_ms": ms,
            "traffic": traffic, "TFLOP/s": tflops, "GB/s": gbs,
            "hbm_frac": gbs / hbm, "tensor_frac": tflops / bf16}
    if t_tensor >= t_hbm:
        base.update({"bound": "tensor", "achieved": tflops, "peak": bf16, "unit": "TFLOP/s",
                     "frac": tflops / bf16})
    else:
        base.update({"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                     "frac": gbs / hbm})
    return base


def measure_secondary(name, args, world, dist):
    """A second workload's step, eager and graph-replayed (no breakdown)."""
    import torch
    cfg = CONFIGS[name]
    rank = dist.get_rank() if dist else 0
    b = Bench(replica_config(cfg, rank), rank)
    for _ in range(args.warmup):
        b.step()
    torch.cuda.synchronize()
    ms = reduce_max(b.timed(b.step, args.steps), dist, "cuda")
    st = int(b.status.item())
    gms = reduce_max(b.graph_timed(args.steps, args.warmup), dist, "cuda")
    b.close()
    del b
    torch.cuda.empty_cache()
    if st:
        raise RuntimeError(f"device status {st} on {name}")
    return {"workload": name, "value": job_value(cfg.T, world, ms), "unit": "tokens/s",
            "ms_per_step": ms, "graph_ms_per_step": gms, "T": cfg.T, "wfmt": cfg.wfmt,
            "slots": cfg.S, "prefilled": cfg.prefill}


def gpu_arm(args, cfg):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist:
            dist.barrier()
        torch.cuda.synchronize()

    from offloaded_expert_slot_gb300 import build
    if rank == 0:
        build.build()
    if dist:
        dist.barrier()
    b = Bench(replica_config(cfg, rank), rank)
    for _ in range(args.warmup):
        b.step()
    torch.cuda.synchronize()
    st = int(b.status.item())
    if st:
        raise RuntimeError(f"device status {st} after warm-up")

    barrier()
    # clocks: sampled from just before the timed region (GPU already under
    # load from these extra untimed steps) to its end
    sampler = ClockSampler(local)
    sampler.start()
    t_end = time.perf_counter() + 0.5
    while time.perf_counter() < t_end:
        b.step()
        torch.cuda.synchronize()
    ms = b.timed(b.step, args.steps)
    clocks = sampler.stop()
    barrier()
    ms_max = reduce_max(ms, dist, "cuda")
    value = job_value(cfg.T, world, ms_max)

    graph_ms = b.graph_timed(args.steps, args.warmup)
    graph_ms = reduce_max(graph_ms, dist, "cuda")

    e2e_ms, bi, bo = b.e2e(args.steps, args.warmup)
    e2e_ms = reduce_max(e2e_ms, dist, "cuda")
    e2e_value = job_value(cfg.T, world, e2e_ms)

    bd, info = b.breakdown(max(3, args.steps // 2))
    link = b.link_probe()
    pk = peaks()
    hbm = float(pk["hbm_gbs"])
    R = cfg.T * cfg.k
    H, I, E = cfg.H, cfg.I, cfg.E
    step_bytes = {
        "route": cfg.T * E * 4 + R * 8,
        "distinct": R * 4 + min(R, E) * 4,
        "align": R * 4 * 2 + info["blocks"] * info["block"] * 4 + info["blocks"] * 4,
        "copy": info["misses"] * cfg.row_bytes,
        "gemm": info["distinct"] * cfg.row_bytes + cfg.T * H * 2 * 2,
    }
    kernels = {}
    for n, b_ in step_bytes.items():
        t_ms = bd[n]
        gbs = b_ / (t_ms / 1e3) / 1e9 if t_ms > 0 else None
        bound_peak = link if n == "copy" else hbm
        kernels[n] = {"ms": round(t_ms, 5), "bytes": b_, "GB/s": gbs,
                      "bound": "host_link" if n == "copy" else "hbm",
                      "frac": (gbs / bound_peak) if gbs else None}
    kernels["ensure"] = {"ms": round(bd["ensure"], 5), "queries": info["queries"],
                         "us_per_query": 1e3 * bd["ensure"] / info["queries"], "bound": "latency"}
    kernels["restore"] = {"ms": round(bd["restore"], 5)}
    dom = max(("route", "distinct", "ensure", "copy", "align", "gemm"), key=lambda n: bd[n])
    tr = TRAFFIC.get(cfg.name, {})
    roof_gemm = gemm_roofline(cfg, info, bd["gemm"], pk, tr.get("gemm_per_step"))
    kernels["gemm"].update({"TFLOP/s": roof_gemm["TFLOP/s"], "tensor_frac": roof_gemm["tensor_frac"],
                            "bound": roof_gemm["bound"]})
    if dom == "copy":
        # the miss copies are bound by the host link, whose peak is probed in
        # this run; the GEMM overlaps them and is reported beside them
        c = kernels["copy"]
        q = info["queries"]
        roofline = {"kernel": "copy_misses_kernel", "bound": "host_link", "achieved": c["GB/s"],
                    "peak": link, "unit": "GB/s", "frac": c["frac"],
                    "traffic": tr.get("copy_per_launch"),
                    "traffic_note": "DRAM read + write per launch from one ncu capture; the rows "
                                    "are read over the host link, and part of a launch's writes "
                                    "is still in L2 when it ends",
                    "peak_source": "measured in this run: 1 GiB pinned host->device cudaMemcpyAsync",
                    "launches": q, "algorithmic_bytes": step_bytes["copy"] / q,
                    "launch_ms": bd["copy"] / q}
    else:
        roofline = roof_gemm
    cpu = cpu_baseline(cfg, b) if rank == 0 else None
    pinned = len(b.src_bufs)
    b.close()
    del b
    torch.cuda.empty_cache()
    secondary = None
    if SECONDARY_CONFIG != cfg.name and not args.no_secondary:
        secondary = measure_secondary(SECONDARY_CONFIG, args, world, dist)
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if cfg.wfmt == "bf16" else "nvfp4-w/f16", "data": "synthetic",
                "config": config_of(cfg, world),
                "step_info": {"queries": info["queries"], "misses_per_step": info["misses"],
                              "distinct": info["distinct"], "block": info["block"],
                              "pinned_source_layers": pinned},
                "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": bi,
                        "d2h_bytes_per_step": bo, "ms_per_step": e2e_ms},
                "gpu_launches": gpu_launches(cfg) * args.steps,
                "graph": {"value": job_value(cfg.T, world, graph_ms), "unit": "tokens/s",
                          "ms_per_step": graph_ms,
                          "what": "the same step captured once as a CUDA graph and replayed"},
                "clocks": clocks, "roofline": roofline, "roofline_gemm": roof_gemm,
                "steps_breakdown": kernels, "host_link_gbs": link, "cpu_baseline": cpu,
                "decode_width": secondary}
        print(json.dumps(line))
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def blas_threads() -> int:
    """Threads of numpy's BLAS pool (the oracle's matrix products; its other
    steps run on one): OPENBLAS_NUM_THREADS as set before numpy loaded."""
    try:
        return max(1, int(os.environ.get("OPENBLAS_NUM_THREADS", CPU_THREADS)))
    except ValueError:
        return CPU_THREADS


def cpu_baseline(cfg, b):
    """The oracle on the host cores over bounded samples (about 10 s)."""
    srcs = [x.numpy() for x in b.src_bufs]
    row = lambda l, e: srcs[b.source_index(l)][e]
    cs, rin = oracle_chunk(cfg, b.rin)
    n_tok = min(cs.T, ORACLE_MLP_TOKENS)
    total, tokens, i = 0.0, 0, 0
    while total < 10.0 and i < 200:
        total += oracle_sample(cs, rin, row, b.prefill, n_tok, 1000 + i)
        tokens += n_tok
        i += 1
    return {"kind": "oracle", "value": tokens / total, "unit": "tokens/s",
            "cores": blas_threads(),
            "sample": f"{i} samples, {total:.1f} s: " + sample_text(cfg, cs, n_tok)}


def sweep(args):
    """Bandwidth sweep of the bookkeeping kernels at sizes where HBM time is
    measurable (beyond the workloads, which are latency-bound): routing of
    65,536 tokens over 512 experts (134 MB of logits) and align of 2^24
    routes.  One JSON line per kernel; not the headline."""
    import torch
    from offloaded_expert_slot_gb300 import build, oes
    build.build()
    oes.load()
    hbm = float(peaks()["hbm_gbs"])
    g = torch.Generator(device="cuda")
    g.manual_seed(7)

    # L2 (129 MB) is flushed before every timed launch by a 256 MB write
    # outside the launch's events, so no input is served from a previous
    # launch's lines (the align's 67 MB of ids would fit)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def timed(fn, steps=20):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for e0, e1 in ev:
            flush.zero_()
            e0.record()
            fn()
            e1.record()
        torch.cuda.synchronize()
        return sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps

    for T, E, k in [(65536, 512, 10), (262144, 512, 8)]:
        logits = torch.randn((T, E), generator=g, device="cuda")
        ids = torch.empty(T * k, dtype=torch.int32, device="cuda")
        w = torch.empty(T * k, dtype=torch.float32, device="cuda")
        ms = timed(lambda: oes.moe_route_topk(logits, T, E, k, ids, w))
        b = T * E * 4 + T * k * 8
        print(json.dumps({"sweep": "moe_route_topk", "T": T, "E": E, "k": k, "ms": ms,
                          "bytes": b, "GB/s": b / ms / 1e6, "hbm_frac": b / ms / 1e6 / hbm,
                          "l2": "flushed before each timed launch"}))
        del logits
    for R, E, B in [(1 << 24, 512, 64), (1 << 24, 2100, 64), (65536, 2100, 64), (40960, 512, 128)]:
        ids = torch.randint(0, E, (R,), generator=g, device="cuda", dtype=torch.int32)
        cap = oes.align_capacity(R, E, B)
        srt = torch.empty(cap, dtype=torch.int32, device="cuda")
        be = torch.empty(cap // B, dtype=torch.int32, device="cuda")
        npp = torch.empty(1, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        wsb = oes.moe_align_workspace_size(R, E, B)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        ms = timed(lambda: oes.moe_align_block_size(ids, R, E, B, 1, srt, be, npp, st, ws, wsb))
        b = R * 4 * 2 + cap * 4 + (cap // B) * 4
        print(json.dumps({"sweep": "moe_align_block_size", "R": R, "E": E, "B": B, "ms": ms,
                          "bytes": b, "GB/s": b / ms / 1e6, "hbm_frac": b / ms / 1e6 / hbm,
                          "l2": "flushed before each timed launch"}))


def crossover(args):
    """Slot path vs staged whole-layer path over a sequence of layers, per
    chunk size: where on-demand loading stops paying (FreeToken PR #676,
    A/B and Known limits; vLLM fork PR #51, Details).  Per chunk size T and
    routing, milliseconds per layer over `n_layers` layers for
      slots      moe_layer_forward_slots per layer (no admission stats), the
                 pool restored to its pre-fill first;
      staged     oes_stage_plan_create (skip resident; one map readback)
                 + moe_layers_forward_staged (next layer copied during this
                 layer's compute) + destroy;
      streamed   the whole layer copied into the staging rows (no skip),
                 with the same prefetch;
      serial     moe_layer_forward_stream per layer (copy, then compute).
    The pool is pre-filled to every slot with seeded keys of all layers, as
    decode would leave it.  One JSON line per (routing, T); not the headline."""
    import torch
    from offloaded_expert_slot_gb300 import build, oes
    from offloaded_expert_slot_gb300.configs import scaled
    from offloaded_expert_slot_gb300.inputs import (empty_slot_row, expert_layer_rows,
                                                    n_source_buffers, pool_prefill,
                                                    router_inputs, source_layer_index)
    build.build()
    oes.load()
    base = CONFIGS[args.config]
    if base.wfmt == "bf16":
        base = scaled(base, L=8, distinct_source_layers=2)
    else:
        # only layers 0..7 are forwarded: 8 distinct sources, the pool's
        # placement still spread over all of the workload's layers
        base = scaled(base, distinct_source_layers=min(base.L, 8))
    base = scaled(base, prefill=base.S)
    n_layers = min(8, base.L)
    E, S, rb = base.E, base.S, base.row_bytes
    srcs = []
    for l in range(n_source_buffers(base)):
        buf = torch.empty((E, rb), dtype=torch.uint8, pin_memory=True)
        expert_layer_rows(base, l, device="cuda", out=buf)
        srcs.append(buf)
    src = oes.oes_expert_source_create([srcs[source_layer_index(base, l)] for l in range(base.L)],
                                       E, rb)
    pool_all = torch.empty((S + 2 * E, rb), dtype=torch.uint8, device="cuda")
    pool = pool_all[:S]
    cache = oes.slot_cache_create(S, base.L, E)
    st = pool_prefill(base)
    oes.slot_cache_load_state(cache, st["slot_key"], st["slot_ts"], st["clock"])
    pool[:] = torch.from_numpy(empty_slot_row(base)).cuda()
    for s_ in np.nonzero(st["slot_key"] >= 0)[0]:
        k_ = int(st["slot_key"][s_])
        pool[int(s_)].copy_(srcs[source_layer_index(base, k_ // E)][k_ % E])
    snap = torch.empty(oes.slot_cache_state_bytes(cache), dtype=torch.uint8, device="cuda")
    oes.slot_cache_snapshot(cache, snap)
    layer_buf = pool_all[S:S + E]
    wfmt = oes.OES_WFMT_BF16 if base.wfmt == "bf16" else oes.OES_WFMT_NVFP4
    desc = oes.layer_desc(E, base.H, base.I, wfmt)
    copy_stream = torch.cuda.Stream()
    layers = list(range(n_layers))
    link = None
    for routing in ("normal", "normal+zipf"):
        best = []
        for T in (8, 16, 32, 64, 128, 256, 384, 512, 768, 1024):
            cfg = scaled(base, T=T, logits=routing, zipf_s=1.1 if routing != "normal" else 0.0)
            rin = router_inputs(cfg)
            x = torch.from_numpy(rin["x"].view(np.int16)).cuda()
            logits = torch.from_numpy(rin["logits"]).cuda()
            wsb = oes.moe_layer_workspace_size(desc, T, cfg.k)
            ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
            out = torch.empty((T, cfg.H), dtype=torch.bfloat16, device="cuda")
            status = torch.zeros(1, dtype=torch.int32, device="cuda")
            ch = oes.chunk(x, T, cfg.k, out, status, ws, wsb, logits=logits)

            def slots():
                oes.slot_cache_restore(cache, snap)
                for l in layers:
                    oes.moe_layer_forward_slots(cache, src, pool, l, desc, ch, 0)

            def staged(skip):
                def run():
                    oes.slot_cache_restore(cache, snap)
                    plan = oes.oes_stage_plan_create(cache, layers, skip)
                    oes.moe_layers_forward_staged(plan, src, pool_all, desc, [ch] * n_layers,
                                                  copy_stream=copy_stream)
                    oes.oes_stage_plan_destroy(plan)
                return run

            def serial():
                for l in layers:
                    oes.moe_layer_forward_stream(src, layer_buf, l, desc, ch,
                                                 copy_stream=copy_stream)

            def timed(fn, steps=3):
                fn()
                torch.cuda.synchronize()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(steps):
                    fn()
                e1.record()
                torch.cuda.synchronize()
                return e0.elapsed_time(e1) / steps / n_layers

            row = {"crossover": base.wfmt, "routing": routing, "T": T, "k": cfg.k, "E": E,
                   "S": S, "n_layers": n_layers,
                   "ms_per_layer": {"slots": timed(slots), "staged": timed(staged(True)),
                                    "streamed": timed(staged(False)), "serial": timed(serial)}}
            assert int(status.item()) == 0
            slots()                                  # the distinct count of the chunk
            torch.cuda.synchronize()
            off = oes.moe_layer_workspace_views(desc, T, cfg.k, ws)["d_count"] - ws.data_ptr()
            row["distinct_experts"] = int(ws[off:off + 4].view(torch.int32).item())
            row["layer_bytes"] = E * rb
            m = row["ms_per_layer"]
            row["faster"] = "slots" if m["slots"] < min(m["staged"], m["streamed"]) else "staged"
            best.append((T, row["faster"]))
            print(json.dumps(row), flush=True)
            del x, logits, ws, out
        cross = next((T for T, f in best if f != "slots"), None)
        print(json.dumps({"crossover_summary": base.wfmt, "routing": routing,
                          "first_T_where_staging_wins": cross}), flush=True)
    oes.slot_cache_destroy(cache)
    oes.oes_expert_source_destroy(src)


def layer_sweep(args):
    """Every layer of the workload forwarded in turn, as a prefill does:
      slots    moe_layer_forward_slots layer after layer (the cache evolves;
               no restore), each layer timed with CUDA events;
      staged   one plan over all layers + moe_layers_forward_staged
               (non-resident runs, next layer copied during this layer);
      serial   moe_layer_forward_stream layer after layer.
    One JSON line with per-layer times of the slot path and the totals; not
    the headline."""
    import torch
    from offloaded_expert_slot_gb300 import build, oes
    from offloaded_expert_slot_gb300.inputs import (empty_slot_row, expert_layer_rows,
                                                    n_source_buffers, pool_prefill,
                                                    router_inputs, source_layer_index)
    build.build()
    oes.load()
    cfg = CONFIGS[args.config]
    E, S, rb, L = cfg.E, cfg.S, cfg.row_bytes, cfg.L
    srcs = []
    for l in range(n_source_buffers(cfg)):
        buf = torch.empty((E, rb), dtype=torch.uint8, pin_memory=True)
        expert_layer_rows(cfg, l, device="cuda", out=buf)
        srcs.append(buf)
    src = oes.oes_expert_source_create([srcs[source_layer_index(cfg, l)] for l in range(L)], E, rb)
    pool_all = torch.empty((S + 2 * E, rb), dtype=torch.uint8, device="cuda")
    pool = pool_all[:S]
    cache = oes.slot_cache_create(S, L, E)

    def reset():
        st = pool_prefill(cfg)
        oes.slot_cache_load_state(cache, st["slot_key"], st["slot_ts"], st["clock"])
        pool[:] = torch.from_numpy(empty_slot_row(cfg)).cuda()
        for s_ in np.nonzero(st["slot_key"] >= 0)[0]:
            k_ = int(st["slot_key"][s_])
            pool[int(s_)].copy_(srcs[source_layer_index(cfg, k_ // E)][k_ % E])
        torch.cuda.synchronize()

    rin = router_inputs(cfg)
    x = torch.from_numpy(rin["x"].view(np.int16)).cuda()
    logits = torch.from_numpy(rin["logits"]).cuda()
    wfmt = oes.OES_WFMT_BF16 if cfg.wfmt == "bf16" else oes.OES_WFMT_NVFP4
    desc = oes.layer_desc(E, cfg.H, cfg.I, wfmt)
    wsb = oes.moe_layer_workspace_size(desc, cfg.T, cfg.k)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    out = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ch = oes.chunk(x, cfg.T, cfg.k, out, status, ws, wsb, logits=logits)
    copy_stream = torch.cuda.Stream()
    layers = list(range(L))

    def ev():
        e = torch.cuda.Event(enable_timing=True)
        e.record()
        return e

    # warm-up: one untimed pass over every layer, so that each pinned source
    # has been read by the GPU once before anything is timed
    reset()
    for l in layers:
        oes.moe_layer_forward_slots(cache, src, pool, l, desc, ch, 0)
    torch.cuda.synchronize()
    reset()
    marks = [ev()]
    for l in layers:
        oes.moe_layer_forward_slots(cache, src, pool, l, desc, ch, 0)
        marks.append(ev())
    torch.cuda.synchronize()
    per_layer = [marks[i].elapsed_time(marks[i + 1]) for i in range(L)]
    reset()
    t0 = ev()
    plan = oes.oes_stage_plan_create(cache, layers, True)
    oes.moe_layers_forward_staged(plan, src, pool_all, desc, [ch] * L, copy_stream=copy_stream)
    t1 = ev()
    torch.cuda.synchronize()
    oes.oes_stage_plan_destroy(plan)
    staged = t0.elapsed_time(t1)
    buf = pool_all[S:S + E]
    t0 = ev()
    for l in layers:
        oes.moe_layer_forward_stream(src, buf, l, desc, ch, copy_stream=copy_stream)
    t1 = ev()
    torch.cuda.synchronize()
    serial = t0.elapsed_time(t1)
    assert int(status.item()) == 0, int(status.item())
    print(json.dumps({"layer_sweep": cfg.name, "layers": L, "T": cfg.T, "k": cfg.k, "E": E,
                      "slots": S, "wfmt": cfg.wfmt,
                      "slots_ms_per_layer": [round(v, 4) for v in per_layer],
                      "slots_total_ms": sum(per_layer),
                      "slots_median_ms": float(np.median(per_layer)),
                      "staged_total_ms": staged, "serial_stream_total_ms": serial,
                      "layer_bytes": E * rb}), flush=True)
    oes.slot_cache_destroy(cache)
    oes.oes_expert_source_destroy(src)


def decode_warm(args):
    """The decode step with a warm cache: every expert the tokens route to is
    already resident (the step is run once before timing and the cache is
    not restored), so the step is routing, the ensures (all hits), align and
    the grouped GEMM over the routed experts -- a weight stream from HBM.
    Per decode width: eager and graph-replayed ms per step, the distinct
    experts, their bytes, and that stream's fraction of the measured HBM
    bandwidth.  One JSON line per width; not the headline."""
    import torch
    from offloaded_expert_slot_gb300 import build, oes
    from offloaded_expert_slot_gb300.configs import scaled
    build.build()
    oes.load()
    hbm = float(peaks()["hbm_gbs"])
    base = CONFIGS[args.config]
    for T in (1, 4, 8, 16, 32, 64):
        cfg = scaled(base, T=T)
        b = Bench(cfg, 0)

        def step():
            oes.moe_layer_forward_slots(b.cache, b.src, b.pool, cfg.layer, b.desc, b.chunk, 1)

        step()                                        # loads the misses: warm from here on
        torch.cuda.synchronize()
        for _ in range(3):
            step()
        ms = b.timed(step, max(args.steps, 20))
        g = torch.cuda.CUDAGraph()
        st = torch.cuda.Stream()
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            with torch.cuda.graph(g, stream=st):
                step()
        torch.cuda.current_stream().wait_stream(st)
        for _ in range(3):
            g.replay()
        gms = b.timed(g.replay, max(args.steps, 20))
        assert int(b.status.item()) == 0, int(b.status.item())
        off = oes.moe_layer_workspace_views(b.desc, T, cfg.k, b.ws)["d_count"] - b.ws.data_ptr()
        D = int(b.ws[off:off + 4].view(torch.int32).item())
        nbytes = D * cfg.row_bytes
        print(json.dumps({"decode_warm": cfg.name, "T": T, "k": cfg.k, "distinct_experts": D,
                          "expert_bytes": nbytes, "ms_eager": ms, "ms_graph": gms,
                          "GB/s_graph": nbytes / gms / 1e6, "hbm_frac_graph": nbytes / gms / 1e6 / hbm,
                          "routed_tokens_per_s_graph": T / gms * 1e3}), flush=True)
        del g
        b.close()
        del b, step
        torch.cuda.empty_cache()


def breakdown_only(args):
    """The per-step breakdown of bench.py's timed step alone: route, distinct,
    each query's ensure and whole-query copy, align and the grouped GEMM as
    separate calls on one stream (the launches the roofline line times), one
    JSON line of per-kernel milliseconds."""
    import torch
    from offloaded_expert_slot_gb300 import build
    build.build()
    cfg = CONFIGS[args.config]
    b = Bench(cfg, 0)
    bd, info = b.breakdown(max(1, args.steps))
    torch.cuda.synchronize()
    print(json.dumps({"breakdown": cfg.name, "ms": bd, **info}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="oes", choices=["oes", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(CONFIGS))
    ap.add_argument("--sweep", action="store_true",
                    help="bandwidth sweep of the routing and align kernels (not the headline)")
    ap.add_argument("--crossover", action="store_true",
                    help="slot path vs staged whole-layer path per chunk size (not the headline)")
    ap.add_argument("--decode-warm", action="store_true",
                    help="decode steps with every routed expert resident (GEMM-bound), per width")
    ap.add_argument("--layers", action="store_true",
                    help="every layer of the workload in turn: slot path, staged, streamed")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the decode-width step measured after the headline")
    ap.add_argument("--breakdown", action="store_true",
                    help="only the per-step breakdown (each step's kernels as separate calls, "
                         "timed with events), for a profiler")
    args = ap.parse_args()
    if args.breakdown:
        breakdown_only(args)
        return
    if args.decode_warm:
        decode_warm(args)
        return
    if args.layers:
        layer_sweep(args)
        return
    if args.crossover:
        crossover(args)
        return
    if args.sweep:
        sweep(args)
        return
    args.warmup = max(args.warmup, 3)
    cfg = CONFIGS[args.config]
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return
        reference_arm(args, cfg)
        return
    gpu_arm(args, cfg)


if __name__ == "__main__":
    main()
