"""Pins for the oracle's NVFP4 activation quantiser (CPU only).

* Hand-computed codes and blocks (tests/golden/nvfp4_act_quant.json): ties
  to even, saturation at 6 and 448, the scale rule, zero blocks.
* e4m3 encoding against torch's float8_e4m3fn cast, an independent
  implementation, on random values and on every midpoint between codes.
* On random blocks every element is within one scale unit, sf * a, of its
  input, and its code is a nearest e2m1 value of v / (sf * a).
* The W4A4 expert MLP stays close to the W4A16 one, and depends on the
  activation scale.
"""
import json
import os

import numpy as np
import pytest
import torch

from conftest import GOLDEN
from oracle.expert_mlp import swiglu_expert, swiglu_expert_w4a4
from oracle.numerics import E2M1_TABLE, E4M3_TABLE
from oracle.quant import e2m1_encode, e4m3_encode_nonneg, quantize_act

G = json.load(open(os.path.join(GOLDEN, "nvfp4_act_quant.json")))


def test_e2m1_hand_codes():
    for x, want in G["e2m1"]:
        got = E2M1_TABLE[e2m1_encode(np.float32(x))]
        assert got == want and np.signbit(got) == np.signbit(want), (x, got, want)


def test_blocks_by_hand():
    for b in G["blocks"]:
        v = np.zeros(16, np.float32)
        v[:len(b["v"])] = b["v"]
        q, sc, deq = quantize_act(v[None], b["a"])
        assert E4M3_TABLE[sc[0, 0]] == b["scale"], b
        assert np.array_equal(deq[0, :len(b["deq"])], np.array(b["deq"])), (b, deq[0])
        assert not deq[0, len(b["deq"]):].any()


def test_e4m3_matches_torch():
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.uniform(0, 448, 20000), np.exp(rng.uniform(-12, 6, 20000))])
    vals = vals[vals <= 448].astype(np.float32)
    mids = ((E4M3_TABLE[:0x7E] + E4M3_TABLE[1:0x7F]) / 2).astype(np.float32)
    for x in (vals, mids):
        ours = E4M3_TABLE[e4m3_encode_nonneg(x)]
        ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
        assert np.array_equal(ours, ref)


@pytest.mark.parametrize("a", [0.37, 1.0, 2.0, 9.0])
def test_random_blocks_bound_and_nearest(a):
    """Blocks whose scale amax / (6 a) is a normal e4m3 number (2^-6 .. 448),
    so that sf is within 1/16 of it and v / (sf a) at most 6.4 in size."""
    rng = np.random.default_rng(int(a * 100))
    v = rng.standard_normal((64, 8, 16))
    target = 6 * a * np.exp(rng.uniform(np.log(2.0 ** -5), np.log(200.0), (64, 8, 1)))
    v = (v * target / np.abs(v).max(axis=-1, keepdims=True)).reshape(64, 128).astype(np.float32)
    q, sc, deq = quantize_act(v, a)
    sf = E4M3_TABLE[sc]                                       # [64, 8]
    unit = np.repeat(sf, 16, axis=1) * np.float32(a)
    assert (np.abs(v - deq * a) <= unit * (1 + 1e-6)).all()
    d = np.repeat((sf.astype(np.float32) * np.float32(a)), 16, axis=1).astype(np.float32)
    r = np.where(d > 0, v / np.where(d > 0, d, 1), 0).astype(np.float64)
    err = np.abs(np.abs(r) - np.abs(E2M1_TABLE[q]))
    best = np.abs(np.abs(r)[..., None] - E2M1_TABLE[:8]).min(axis=-1)
    assert np.allclose(err, best, rtol=0, atol=1e-12)


def test_scale_underflow_gives_a_zero_block():
    """A block whose amax / (6 a) rounds to e4m3 zero (below 2^-10) is all
    zero; just above, the smallest subnormal scale 2^-9 is used."""
    a = 9.0
    v = np.zeros((1, 16), np.float32)
    v[0, 0] = np.float32(6 * a * 2.0 ** -11)
    q, sc, deq = quantize_act(v, a)
    assert sc[0, 0] == 0 and not deq.any()
    v[0, 0] = np.float32(6 * a * 2.0 ** -9)
    q, sc, deq = quantize_act(v, a)
    assert E4M3_TABLE[sc[0, 0]] == 2.0 ** -9 and deq[0, 0] == 6 * 2.0 ** -9


def test_w4a4_mlp_close_to_w4a16_and_scale_dependent():
    rng = np.random.default_rng(1)
    H, I = 64, 32
    x = rng.standard_normal((5, H)).astype(np.float32).astype(np.float64)
    w13 = rng.standard_normal((2 * I, H)) * 0.05
    w2 = rng.standard_normal((H, I)) * 0.05
    y16 = swiglu_expert(x, w13, w2)
    y4 = swiglu_expert_w4a4(x, w13, w2, 2.0, 3.0)
    rel = np.linalg.norm(y4 - y16) / np.linalg.norm(y16)
    assert 0 < rel < 0.25
    assert not np.array_equal(y4, swiglu_expert_w4a4(x, w13, w2, 9.0, 3.0))
