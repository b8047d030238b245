"""GPU parity: routing, distinct experts and moe_align_block_size against the
oracle, bit-exact for ids, distinct lists and align outputs; router
weights within 2e-6 relative (expf in fp32 against fp64)."""
import numpy as np
import pytest
import torch

from gpu_util import bits16, cuda, f32, i32, lib, scratch, status
from offloaded_expert_slot_gb300 import oes
from offloaded_expert_slot_gb300.configs import C1, C2, C3, C4, C5, C5B
from offloaded_expert_slot_gb300.inputs import router_inputs, uniform_routes
from oracle.align import moe_align_block_size as oracle_align
from oracle.distinct import distinct_experts
from oracle.router import gate_logits, route_topk, route_topk_bf16

pytestmark = pytest.mark.gpu


def gpu_route(logits: np.ndarray, k: int):
    T, E = logits.shape
    ids, w = i32(T * k), f32(T * k)
    oes.moe_route_topk(cuda(logits), T, E, k, ids, w)
    torch.cuda.synchronize()
    return ids.cpu().numpy().reshape(T, k), w.cpu().numpy().reshape(T, k)


@pytest.mark.parametrize("cfg", [C2, C3, C4, C5], ids=lambda c: c.name)
def test_topk_matches_oracle(cfg):
    lib()
    logits = router_inputs(cfg)["logits"]
    ids, w = gpu_route(logits, cfg.k)
    rows = np.arange(cfg.T) if cfg.T <= 600 else np.random.default_rng(0).choice(cfg.T, 600, False)
    oids, ow = route_topk(logits[rows], cfg.k)
    assert np.array_equal(ids[rows], oids)
    np.testing.assert_allclose(w[rows], ow, rtol=2e-6, atol=1e-7)


def test_topk_ties_and_wide_experts():
    lib()
    g = np.random.default_rng(11)
    for E, k in [(8, 2), (64, 8), (512, 10), (2100, 32), (4096, 16)]:
        logits = (g.integers(-4, 5, size=(33, E)) * 0.25).astype(np.float32)   # many ties
        ids, w = gpu_route(logits, k)
        oids, ow = route_topk(logits, k)
        assert np.array_equal(ids, oids), E
        np.testing.assert_allclose(w, ow, rtol=2e-6, atol=1e-7)


def test_topk_signed_zeros_infinities_and_k16():
    """The per-logit ordering the kernel keys on: -0 ties with +0 (lower id
    first), -inf ranks below every finite logit and gets weight 0; and k = 16
    on 512 and 33 experts."""
    lib()
    g = np.random.default_rng(12)
    for E, k in [(512, 10), (512, 16), (33, 16), (33, 3)]:
        vals = np.array([-np.inf, -0.0, 0.0, -1.0, 0.5, 2.0], dtype=np.float32)
        logits = vals[g.integers(0, len(vals), size=(40, E))]
        logits[::3] = g.standard_normal((logits[::3].shape[0], E)).astype(np.float32)
        logits[1] = -np.inf                      # fewer finite logits than k: -inf ones
        logits[1, g.choice(E, 2, replace=False)] = [1.0, -0.0]   # are taken in id order
        ids, w = gpu_route(logits, k)
        oids, ow = route_topk(logits, k)
        assert np.array_equal(ids, oids), (E, k)
        np.testing.assert_allclose(w, ow, rtol=2e-6, atol=1e-7)


def test_topk_nan_logits_rank_as_minus_infinity():
    """NaN logits (the router's reading: NaN ranks as -inf) mixed with -inf
    and finite ones, including rows with fewer than k finite logits: ids and
    weights against the oracle."""
    lib()
    g = np.random.default_rng(14)
    for E, k in [(512, 10), (33, 16), (2100, 32)]:
        logits = g.standard_normal((24, E)).astype(np.float32)
        logits[g.random((24, E)) < 0.2] = np.nan
        logits[g.random((24, E)) < 0.1] = -np.inf
        logits[2] = np.nan
        logits[2, :3] = [1.0, -np.inf, 0.5]
        ids, w = gpu_route(logits, k)
        oids, ow = route_topk(logits, k)
        assert np.array_equal(ids, oids), (E, k)
        np.testing.assert_allclose(w, ow, rtol=2e-6, atol=1e-7)


def test_topk_bf16_logits():
    """bf16 logits route as their exact fp32 widening: ids bit-exact against
    the oracle, weights within its bound, and both identical bit for bit to the
    fp32 call on the widened values.  Truncated normals give many ties; -inf
    and -0 are mixed in.  One case passes a torch.bfloat16 tensor."""
    lib()
    g = np.random.default_rng(13)
    for E, k in [(8, 2), (33, 16), (512, 10), (2100, 32), (4096, 8)]:
        f = g.standard_normal((37, E)).astype(np.float32)
        bits = (f.view(np.uint32) >> 16).astype(np.uint16)
        bits[::5, ::7] = 0xff80
        bits[1::5, ::3] = 0x8000
        T = bits.shape[0]
        ids, w = i32(T * k), f32(T * k)
        dev = bits16(bits)
        if E == 512:
            oes.moe_route_topk(dev.view(torch.bfloat16), T, E, k, ids, w)
        else:
            oes.moe_route_topk(dev, T, E, k, ids, w, dtype=oes.OES_LOGITS_BF16)
        torch.cuda.synchronize()
        gi, gw = ids.cpu().numpy().reshape(T, k), w.cpu().numpy().reshape(T, k)
        oids, ow = route_topk_bf16(bits, k)
        assert np.array_equal(gi, oids), (E, k)
        np.testing.assert_allclose(gw, ow, rtol=2e-6, atol=1e-7)
        wide = (bits.astype(np.uint32) << 16).view(np.float32)
        fi, fw = gpu_route(wide, k)
        assert np.array_equal(gi, fi) and np.array_equal(gw.view(np.uint32), fw.view(np.uint32))


def _filter_rows(g, E, k, V, n_rand):
    """Rows around the threshold filter's edges for a lane layout of V logits a
    load: c copies of the top value spread over distinct lanes (c candidates
    exactly once c >= k: 31, 32 fit, 33 and 40 take the fallback), fewer than k
    copies, one lane's entries all equal, -inf below k finite lanes, signed
    zeros at the threshold, then random rows whose ties straddle it."""
    rows = []
    spread = lambda c: (V * (np.arange(c) % 32) + 32 * V * (np.arange(c) // 32)) % E
    for c in (1, k - 1, k, k + 1, 31, 32, 33, 40):
        r = np.minimum(g.standard_normal(E), 1.0).astype(np.float32)
        r[spread(c)] = 3.5
        rows.append(r)
    r = np.minimum(g.standard_normal(E), 1.0).astype(np.float32)
    lane0 = (np.arange(E) // V) % 32 == 0
    r[lane0] = 2.0
    rows.append(r)
    r = np.full(E, -np.inf, np.float32)
    r[spread(k - 1)] = g.standard_normal(k - 1)
    rows.append(r)
    r = np.minimum(g.standard_normal(E), -1.0).astype(np.float32)
    r[spread(2 * k)] = np.where(np.arange(2 * k) % 2, 0.0, -0.0)
    rows.append(r)
    for _ in range(n_rand):
        r = np.minimum(g.standard_normal(E), 1.0).astype(np.float32)
        for val, hi in ((3.0, k + 2), (2.0, 40), (1.5, 40)):
            r[g.choice(E, g.integers(0, min(hi, E)), replace=False)] = val
        if g.random() < 0.2:
            r[g.random(E) < 0.1] = np.nan
        rows.append(r)
    return np.stack(rows)


def test_topk_threshold_filter_edges():
    """The threshold-filter top-k (rows of at most 1024 experts, 16-byte
    aligned, E a multiple of the load width) on rows built around its edges:
    ids bit-exact against the oracle and weights within its bound; and the
    same rows through an unaligned pointer, which takes the round-based
    kernel, give the same ids and the same weights bit for bit."""
    lib()
    g = np.random.default_rng(15)
    for E, k in [(512, 10), (512, 8), (512, 16), (128, 10), (200, 10), (1024, 10), (96, 20),
                 (64, 32), (4, 2)]:
        logits = _filter_rows(g, E, k, 4, 150)
        T = logits.shape[0]
        ids, w = gpu_route(logits, k)
        oids, ow = route_topk(logits, k)
        assert np.array_equal(ids, oids), (E, k)
        np.testing.assert_allclose(w, ow, rtol=2e-6, atol=1e-7)
        buf = torch.zeros(T * E + 1, dtype=torch.float32, device="cuda")
        buf[1:] = cuda(logits).reshape(-1)
        ui, uw = i32(T * k), f32(T * k)
        oes.moe_route_topk(buf[1:], T, E, k, ui, uw)
        torch.cuda.synchronize()
        assert np.array_equal(ui.cpu().numpy().reshape(T, k), ids), (E, k)
        assert np.array_equal(uw.cpu().numpy().view(np.uint32).reshape(T, k), w.view(np.uint32)), (E, k)
    for E, k in [(512, 10), (256, 8), (1024, 16), (8, 2)]:
        f = _filter_rows(g, E, k, 8, 100)
        bits = (f.view(np.uint32) >> 16).astype(np.uint16)
        T = bits.shape[0]
        ids, w = i32(T * k), f32(T * k)
        oes.moe_route_topk(bits16(bits), T, E, k, ids, w, dtype=oes.OES_LOGITS_BF16)
        torch.cuda.synchronize()
        gi, gw = ids.cpu().numpy().reshape(T, k), w.cpu().numpy().reshape(T, k)
        oids, ow = route_topk_bf16(bits, k)
        assert np.array_equal(gi, oids), (E, k)
        np.testing.assert_allclose(gw, ow, rtol=2e-6, atol=1e-7)


def test_gate_logits_tiny_workload():
    """The tiny workload's router: bf16 gate, fp32 sums; the top-2 decision
    is compared where its margin exceeds the fp32 rounding of the sums."""
    lib()
    rin = router_inputs(C1)
    logits = torch.zeros(C1.T * C1.E, dtype=torch.float32, device="cuda")
    oes.moe_gate_logits(bits16(rin["x"]), bits16(rin["gate"]), C1.T, C1.H, C1.E, logits)
    torch.cuda.synchronize()
    got = logits.cpu().numpy().reshape(C1.T, C1.E)
    want = gate_logits(rin["x"], rin["gate"])
    np.testing.assert_allclose(got, want, rtol=1e-5, atol=1e-6)
    srt = np.sort(want, axis=1)
    assert (srt[:, -C1.k] - srt[:, -C1.k - 1]).min() > 1e-4
    ids, _ = gpu_route(got, C1.k)
    oids, _ = route_topk(want, C1.k)
    assert np.array_equal(ids, oids)


@pytest.mark.parametrize("R,E", [(0, 8), (1, 1), (32, 8), (320, 512), (2000, 512), (40960, 512),
                                 (65536, 2100), (5000, 4096)])
def test_distinct_matches_oracle(R, E):
    lib()
    g = np.random.default_rng(R + E)
    ids = g.integers(-1, E, size=R).astype(np.int32)
    n = min(R, E)
    d, cnt = i32(n, 7), i32(1, 7)
    oes.moe_distinct_experts(cuda(ids) if R else 0, R, E, d if n else 0, cnt)
    torch.cuda.synchronize()
    od, oD = distinct_experts(ids, E)
    assert int(cnt.item()) == oD
    assert np.array_equal(d.cpu().numpy()[:n], od)


def gpu_align(ids: np.ndarray, E: int, B: int, ignore_invalid=True):
    R = ids.size
    cap = oes.align_capacity(R, E, B)
    s, b, n, st = i32(cap, -7), i32(cap // B, -7), i32(1, -7), status()
    wsb = oes.moe_align_workspace_size(R, E, B)
    ws = scratch(wsb)
    oes.moe_align_block_size(cuda(ids.astype(np.int32)) if R else 0, R, E, B, ignore_invalid,
                             s if cap else 0, b if cap else 0, n, st, ws, ws.numel())
    torch.cuda.synchronize()
    return s.cpu().numpy()[:cap], b.cpu().numpy()[:cap // B], int(n.item()), int(st.item())


def _routes_of(cfg):
    ids, _ = route_topk(router_inputs(cfg)["logits"], cfg.k)    # the oracle's routing
    return ids.reshape(-1)


@pytest.mark.parametrize("cfg", [C2, C3, C4, C5], ids=lambda c: c.name)
def test_align_workload_sizes(cfg):
    lib()
    ids = _routes_of(cfg)
    B = oes.oes_tile_plan(ids.size, cfg.E)
    s, b, n, st = gpu_align(ids, cfg.E, B)
    os_, ob, on, _ = oracle_align(ids, cfg.E, B)
    assert n == on and st == 0
    assert np.array_equal(s, os_) and np.array_equal(b, ob)


@pytest.mark.parametrize("E", list(C5B.Es) + [1024, 4096])
def test_align_past_1024_experts(E):
    """FreeToken PR #676, Tests: 8192 tokens x top-8 uniformly routed at 1023
    and 2100 experts, block 64: each route exactly once, inside a block of
    its own expert -- here bit-exact against the oracle."""
    lib()
    ids = uniform_routes(C5B.T, C5B.k, E, C5B.seed)
    s, b, n, st = gpu_align(ids, E, C5B.block)
    os_, ob, on, _ = oracle_align(ids, E, C5B.block)
    assert n == on and st == 0
    assert np.array_equal(s, os_) and np.array_equal(b, ob)


@pytest.mark.parametrize("R,E,B", [(0, 5, 4), (1, 1, 1), (7, 3, 1), (100, 7, 3), (999, 64, 16),
                                   (1024, 2100, 16), (1025, 2100, 16), (1000, 4096, 128),
                                   (3000, 1, 128), (4099, 4096, 16)])
def test_align_edges_and_invalid_ids(R, E, B):
    lib()
    g = np.random.default_rng(R * 7 + E)
    ids = g.integers(-2, E + 2, size=R)
    for ignore in (True, False):
        s, b, n, st = gpu_align(ids, E, B, ignore_invalid=ignore)
        os_, ob, on, bad = oracle_align(ids, E, B, ignore_invalid=ignore)
        assert n == on
        assert np.array_equal(s, os_) and np.array_equal(b, ob)
        assert (st == oes.OES_DEV_BAD_ID) == bad


def _stable_sort_layout(ids: np.ndarray, E: int, B: int):
    """The align's definition written with numpy's stable argsort: routes of
    each expert in ascending order, each expert padded to a multiple of B with
    the value R, block b holding its expert (-1 past the last block)."""
    R = ids.size
    cnt = np.bincount(ids, minlength=E).astype(np.int64)
    padded = (cnt + B - 1) // B * B
    off = np.concatenate([[0], np.cumsum(padded)[:-1]])
    cap = oes.align_capacity(R, E, B)
    s = np.full(cap, R, dtype=np.int32)
    order = np.argsort(ids, kind="stable").astype(np.int32)
    starts = np.concatenate([[0], np.cumsum(cnt)[:-1]])
    pos = off[ids[order]] + (np.arange(R) - starts[ids[order]])
    s[pos] = order
    be = np.full(cap // B, -1, dtype=np.int32)
    for e in np.nonzero(padded)[0]:
        be[off[e] // B:(off[e] + padded[e]) // B] = e
    return s, be, int(padded.sum())


def test_align_large_chunk_count():
    """2^25 + 123 routes over 600 experts: about two thousand CTA ranges, so
    the per-CTA counts are scanned over several bands, each CTA's routes are
    ordered in shared memory and written as runs; bit-exact against the
    stable-sort definition."""
    lib()
    R, E, B = (1 << 25) + 123, 600, 64
    ids = np.random.default_rng(21).integers(0, E, size=R).astype(np.int32)
    s, b, n, st = gpu_align(ids, E, B)
    ws, wb, wn = _stable_sort_layout(ids, E, B)
    assert st == 0 and n == wn
    assert np.array_equal(b, wb)
    assert np.array_equal(s, ws)
