"""GPU parity of the W4A4 NVFP4 path (activations quantised under the max of
the layer's input scales, FreeToken PR #676, Solution and Tests), through
the C ABI.

* x quantised per 16 along H: the GEMM's f16 copy equals the oracle's
  q * sf bit for bit under the layer's scale (2.0 or 3.0), and differs from
  what the other slots' 9.0 would give.
* h quantised per 16 along I in GEMM1's epilogue: every code is checked
  against the oracle's fp64 h (w4a4_check.py): it must be the oracle's code
  wherever the fp32 bound on the GPU's h leaves one code possible, and may
  differ by one step only where that bound straddles a rounding boundary;
  on the weight-major and the token-major kernels, and at the NVFP4
  workload's shape (600 tokens x top-10 over 512 experts, hidden 2048,
  intermediate 768, the layer's scale 2.0 against the other slots' 9.0).
* Layer output vs the oracle within the NVFP4 tolerance; the slot path
  equals the streamed path byte for byte, also at the workload's shape.
"""
import numpy as np
import pytest
import torch

from gpu_util import Workload, cuda, i32, lib, scratch, status
from offloaded_expert_slot_gb300 import oes
from offloaded_expert_slot_gb300.configs import C4, scaled
from oracle.expert_mlp import expert_weights
from oracle.layer import forward_slots, forward_stream, route
from oracle.numerics import bf16_to_f64 as obf16
from oracle.quant import quantize_act
from oracle.slot_cache import SlotCache
from test_gpu_layer import check_close
from w4a4_check import check_codes, h_with_bound

pytestmark = pytest.mark.gpu

W4A4_TM = scaled(C4, name="w4a4_token_major", T=96, k=4, E=16, H=256, I=192, S=40, L=2, prefill=20,
                 w4a4=True)
W4A4_WM = scaled(C4, name="w4a4_weight_major", T=40, k=3, E=16, H=256, I=192, S=40, L=2,
                 prefill=20, w4a4=True)
# the NVFP4 workload's own shape and scales, W4A4
W4A4_C4 = scaled(C4, name="w4a4_nvfp4_prefill", w4a4=True)
C4_SAMPLED_TOKENS = 32


def f16_values(t: torch.Tensor) -> np.ndarray:
    # workspace regions include padding rows no kernel writes (any bits)
    with np.errstate(invalid="ignore"):
        return t.cpu().numpy().view(np.float16).astype(np.float64)


@pytest.mark.parametrize("cfg", [W4A4_TM, W4A4_WM, W4A4_C4], ids=lambda c: c.name)
def test_w4a4_gemm_steps(cfg):
    lib()
    full = cfg is W4A4_C4
    w = Workload(cfg, gen_device="cuda" if full else "cpu")
    T, k, E, H, I = cfg.T, cfg.k, cfg.E, cfg.H, cfg.I
    R = T * k
    layer = cfg.layer
    a = cfg.layer_input_scales[layer]
    # the streamed layout: the layer's rows in one buffer, identity remap
    buf = torch.empty((E, cfg.row_bytes), dtype=torch.uint8, device="cuda")
    oes.oes_copy_layer(w.src, layer, buf)
    e2s = cuda(np.arange(E, dtype=np.int32))
    s13 = torch.full((E,), a, dtype=torch.float32, device="cuda")
    view = oes.routed_experts(layer, E, e2s, oes.OES_WFMT_NVFP4_W4A4, buf, cfg.row_bytes, E, H, I,
                              s13, s13)
    ids, wts = i32(R), torch.empty(R, dtype=torch.float32, device="cuda")
    oes.moe_route_topk(w.logits, T, E, k, ids, wts)
    B = oes.oes_tile_plan(R, E)
    assert B == (16 if cfg is W4A4_WM else 128)
    cap = oes.align_capacity(R, E, B)
    srt, be, npp, st = i32(cap), i32(cap // B), i32(1), status()
    awsb = oes.moe_align_workspace_size(R, E, B)
    aws = scratch(awsb)
    oes.moe_align_block_size(ids, R, E, B, 1, srt, be, npp, st, aws, awsb)
    gwsb = oes.moe_grouped_gemm_workspace_size(view, T, k)
    gws = scratch(gwsb)
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    oes.moe_grouped_gemm_slots(view, w.x, T, k, ids, wts, srt, be, npp, B, gws, gwsb, out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    v = oes.moe_grouped_gemm_workspace_views(view, T, k, gws)
    base = gws.data_ptr()

    def region(ptr, n):
        return gws[ptr - base:ptr - base + 2 * n]

    # x: bit for bit under the layer's scale, and not under 9.0
    x32 = obf16(w.rin["x"]).astype(np.float32)
    x16 = f16_values(region(v["x16"], T * H)).reshape(T, H)
    assert np.array_equal(x16, quantize_act(x32, a)[2])
    assert not np.array_equal(x16, quantize_act(x32, 9.0)[2])

    # h: every code of the checked routes against the oracle's fp64 h
    _l, oids, _w = route(w.rin, k)
    assert np.array_equal(ids.cpu().numpy().reshape(T, k), oids)
    sorted_ids = srt.cpu().numpy()
    h_gpu = f16_values(region(v["h"], cap * I)).reshape(cap, I)
    xq = quantize_act(x32, a)[2] * a
    toks = (np.random.default_rng(8).choice(T, C4_SAMPLED_TOKENS, replace=False) if full
            else np.arange(T))
    want_tok = np.zeros(T, bool)
    want_tok[toks] = True
    by_expert = {}
    for p in range(int(npp.item())):
        r = int(sorted_ids[p])
        if r < R and want_tok[r // k]:
            by_expert.setdefault(int(oids.reshape(-1)[r]), []).append((p, r))
    g_rows, h_rows, d_rows = [], [], []
    for e, prs in sorted(by_expert.items()):
        w13, _w2 = expert_weights(w.source_row(layer, e), "nvfp4", H, I)
        h, dh = h_with_bound(xq[[r // k for _p, r in prs]], w13, I)
        g_rows.append(h_gpu[[p for p, _r in prs]])
        h_rows.append(h)
        d_rows.append(dh)
    bad, differ, total = check_codes(np.concatenate(g_rows), np.concatenate(h_rows),
                                     np.concatenate(d_rows), a)
    assert total == len(toks) * k * I
    assert bad == [], (bad[:10], len(bad), differ, total)
    assert differ <= 0.01 * total, (differ, total)

    rows = toks if full else None
    o = forward_stream(cfg, w.rin, lambda e: w.source_row(layer, e), block=B,
                       tokens=toks if full else None)
    check_close(out, o["out"], "nvfp4", rows)
    w.close()


@pytest.mark.parametrize("cfg", [scaled(W4A4_TM, layer=1), W4A4_C4], ids=["medium_layer1", "nvfp4_prefill"])
def test_w4a4_layer_slot_equals_stream_and_oracle(cfg):
    lib()
    full = cfg is W4A4_C4
    w = Workload(cfg, gen_device="cuda" if full else "cpu")
    layer = cfg.layer
    a = cfg.layer_input_scales[layer]
    s13 = torch.full((cfg.E,), a, dtype=torch.float32, device="cuda")
    desc = oes.layer_desc(cfg.E, cfg.H, cfg.I, oes.OES_WFMT_NVFP4_W4A4, s13, s13)
    outs = []
    for path in ("slots", "stream"):
        wsb = oes.moe_layer_workspace_size(desc, cfg.T, cfg.k)
        ws = scratch(wsb)
        out = torch.zeros((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
        st = status()
        ch = oes.chunk(w.x, cfg.T, cfg.k, out, st, ws, wsb, logits=w.logits)
        if path == "slots":
            oes.moe_layer_forward_slots(w.cache, w.src, w.pool, layer, desc, ch, 0)
        else:
            buf = torch.empty((cfg.E, cfg.row_bytes), dtype=torch.uint8, device="cuda")
            oes.moe_layer_forward_stream(w.src, buf, layer, desc, ch,
                                         copy_stream=torch.cuda.Stream())
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    st0 = w.prefill
    ocache = SlotCache.from_state(cfg.S, cfg.L, cfg.E, st0["slot_key"], st0["slot_ts"], st0["clock"])
    toks = np.random.default_rng(9).choice(cfg.T, 24, replace=False) if full else None
    o = forward_slots(cfg, w.rin, w.source_row, ocache, w.oracle_pool(),
                      block=oes.oes_tile_plan(cfg.T * cfg.k, cfg.E), layer=layer, tokens=toks)
    check_close(outs[0], o["out"], "nvfp4", toks)
    now = oes.slot_cache_read_state(w.cache, cfg.S, cfg.L, cfg.E)
    assert np.array_equal(now["slot_key"], ocache.slot_key)
    assert np.array_equal(now["map"], ocache.map)
    w.close()


def test_w4a4_needs_the_layer_scales():
    lib()
    cfg = W4A4_WM
    view = oes.routed_experts(0, cfg.E, 16, oes.OES_WFMT_NVFP4_W4A4, 256, cfg.row_bytes, cfg.E,
                              cfg.H, cfg.I)
    with pytest.raises(oes.OesError) as e:
        oes.moe_grouped_gemm_slots(view, 256, cfg.T, cfg.k, 16, 16, 16, 16, 16, 16, 256, 1 << 30,
                                   256, 16, stream=0)
    assert e.value.code == oes.OES_ERR_INVALID_ARG


def test_refused_gemm_leaves_the_cache_unchanged():
    """A W4A4 layer handed without its input scales is refused before the
    slot path launches anything: no ensure runs, so the tables still match
    the pool's bytes."""
    lib()
    cfg = W4A4_WM
    w = Workload(cfg, gen_device="cpu")
    before = oes.slot_cache_read_state(w.cache, cfg.S, cfg.L, cfg.E)
    desc = oes.layer_desc(cfg.E, cfg.H, cfg.I, oes.OES_WFMT_NVFP4_W4A4)
    wsb = oes.moe_layer_workspace_size(desc, cfg.T, cfg.k)
    ws = scratch(wsb)
    out = torch.zeros((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
    st = status()
    ch = oes.chunk(w.x, cfg.T, cfg.k, out, st, ws, wsb, logits=w.logits)
    with pytest.raises(oes.OesError) as e:
        oes.moe_layer_forward_slots(w.cache, w.src, w.pool, 0, desc, ch, 1)
    assert e.value.code == oes.OES_ERR_INVALID_ARG
    torch.cuda.synchronize()
    after = oes.slot_cache_read_state(w.cache, cfg.S, cfg.L, cfg.E)
    for key in ("map", "slot_key", "slot_ts", "clock", "hits", "misses"):
        assert np.array_equal(np.asarray(after[key]), np.asarray(before[key])), key
    w.close()
