"""The W4A4 code checker itself, on the CPU: it must accept the oracle's own
codes and a one-step move at a boundary the fp32 bound straddles, and
refuse a move away from any boundary, a two-step move, a wrong block
scale, and a value off the e2m1 grid."""
import numpy as np

from oracle.quant import quantize_act
from w4a4_check import check_codes, h_with_bound


def _case(seed=0, n=6, K=256, I=64):
    g = np.random.default_rng(seed)
    xq = quantize_act(g.standard_normal((n, K)).astype(np.float32), 2.0)[2] * 2.0
    w13 = g.standard_normal((2 * I, K)) * 0.02
    h, dh = h_with_bound(xq, w13, I)
    return h, dh


def test_the_oracles_own_codes_pass():
    h, dh = _case()
    want = quantize_act(h.astype(np.float32), 3.0)[2]
    bad, differ, total = check_codes(want, h, dh, 3.0)
    assert bad == [] and differ == 0 and total == h.size


def test_bound_is_small_but_positive():
    h, dh = _case(1)
    assert (dh > 0).all()
    assert np.median(dh / np.maximum(np.abs(h), 1e-12)) < 1e-3


def _boundary_case(a=3.0):
    """One block whose element 3 sits exactly at the 1.25 midpoint between
    codes 1.0 and 1.5, relative to a scale fixed by element 0 (= 6 sf a)."""
    sf = 0.5
    h = np.zeros(16)
    h[0] = 6 * sf * a                 # amax: the block scale is exactly sf
    h[3] = 1.25 * sf * a              # a tie: the oracle rounds it to even (1.0)
    h[5] = 2.9 * sf * a               # far from any boundary: code 3.0
    dh = np.full(16, 1e-6)
    return h[None], dh[None], sf, a


def test_one_step_move_at_a_straddled_boundary_passes():
    h, dh, sf, a = _boundary_case()
    want = quantize_act(h.astype(np.float32), a)[2]
    assert want[0, 3] == 1.0 * sf
    got = want.copy()
    got[0, 3] = 1.5 * sf              # the other side of the boundary
    bad, differ, _ = check_codes(got, h, dh, a)
    assert bad == [] and differ == 1


def test_move_away_from_a_boundary_fails():
    h, dh, sf, a = _boundary_case()
    got = quantize_act(h.astype(np.float32), a)[2].copy()
    got[0, 5] = 4.0 * sf              # 2.9 is nowhere near the 3/4 boundary
    bad, _, _ = check_codes(got, h, dh, a)
    assert bad == [(0, 0)]


def test_two_step_move_fails():
    h, dh, sf, a = _boundary_case()
    got = quantize_act(h.astype(np.float32), a)[2].copy()
    got[0, 3] = 2.0 * sf              # two codes past the 1.0/1.5 boundary
    bad, _, _ = check_codes(got, h, dh, a)
    assert bad == [(0, 0)]


def test_wrong_block_scale_fails():
    h, dh, sf, a = _boundary_case()
    got = quantize_act(h.astype(np.float32), a)[2] * 2.0     # every code under twice the scale
    bad, _, _ = check_codes(got, h, dh, a)
    assert bad == [(0, 0)]


def test_value_off_the_grid_fails():
    h, dh, sf, a = _boundary_case()
    got = quantize_act(h.astype(np.float32), a)[2].copy()
    got[0, 5] = 2.75 * sf
    bad, _, _ = check_codes(got, h, dh, a)
    assert bad == [(0, 0)]
