"""Pins for the oracle's expert MLP, NVFP4 decoding and combine (CPU only)."""
import json
import math
import os

import numpy as np
import pytest
import torch

from conftest import GOLDEN
from oracle.expert_mlp import combine, expert_weights, input_scales, swiglu_expert
from oracle.numerics import E2M1_TABLE, E4M3_TABLE, decode_e2m1_packed
from offloaded_expert_slot_gb300.configs import C1, expert_row_bytes, nvfp4_offsets, scaled
from offloaded_expert_slot_gb300.inputs import expert_layer_rows, f32_to_bf16_bits


def test_nvfp4_codes_golden():
    g = json.load(open(os.path.join(GOLDEN, "nvfp4_codes.json")))
    assert E2M1_TABLE.tolist() == g["e2m1"]
    assert all(math.copysign(1, a) == math.copysign(1, b) for a, b in zip(E2M1_TABLE, g["e2m1"]))
    for code, val in g["e4m3"].items():
        assert E4M3_TABLE[int(code)] == val


def test_e4m3_matches_torch_float8():
    """Every e4m3 code against torch's float8_e4m3fn widening (a library routine)."""
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    ref = ref.numpy()
    both_nan = np.isnan(ref) & np.isnan(E4M3_TABLE)
    assert np.array_equal(ref[~both_nan], E4M3_TABLE[~both_nan])
    assert both_nan.sum() == 2


def test_e2m1_nibble_order():
    packed = np.array([[0x71, 0xF2]], dtype=np.uint8)    # elements 0x1, 0x7, 0x2, 0xF
    assert decode_e2m1_packed(packed, 4).tolist() == [[0.5, 6.0, 1.0, -6.0]]


def test_swiglu_closed_form():
    """H = I = 2 with exact inputs; the value is worked out by hand:
    g = (2, -1), u = (0.25, 3), h_i = g_i / (1 + e^-g_i) * u_i, y = w2 @ h.
    Swapping gate and up, dropping the sigmoid's sign or transposing w2
    changes the result."""
    x = np.array([[1.0, 2.0]])
    w13 = np.array([[1.0, 0.5], [0.0, -0.5], [0.25, 0.0], [1.0, 1.0]])
    w2 = np.array([[1.0, 2.0], [-1.0, 0.5]])
    h0 = 2.0 / (1.0 + math.exp(-2.0)) * 0.25
    h1 = -1.0 / (1.0 + math.exp(1.0)) * 3.0
    want = [h0 + 2.0 * h1, -h0 + 0.5 * h1]
    np.testing.assert_allclose(swiglu_expert(x, w13, w2)[0], want, rtol=1e-15)
    assert abs(want[0] - (-1.1732499892310294)) < 1e-15
    assert abs(want[1] - (-0.8438106710439339)) < 1e-15


def test_swiglu_large_gate_is_linear():
    """silu(g) -> g for large g and -> 0 for very negative g: the MLP becomes
    w2 @ (g * u) or 0."""
    x = np.array([[1.0]])
    w13 = np.array([[60.0], [0.5]])          # gate 60, up 0.5
    w2 = np.array([[2.0]])
    np.testing.assert_allclose(swiglu_expert(x, w13, w2), [[60.0 * 0.5 * 2.0]], rtol=1e-12)
    w13n = np.array([[-60.0], [0.5]])
    assert abs(swiglu_expert(x, w13n, w2)[0, 0]) < 1e-20


def test_combine_closed_form():
    T, k, H = 3, 2, 4
    y = np.arange(T * k * H, dtype=np.float64).reshape(T * k, H)
    w = np.array([[0.25, 0.75], [1.0, 0.0], [0.5, 0.5]], dtype=np.float32)
    out = combine(y, w, T, k)
    for t in range(T):
        np.testing.assert_array_equal(out[t], 0.25 * y[2 * t] + 0.75 * y[2 * t + 1] if t == 0 else
                                      (y[2] if t == 1 else 0.5 * (y[4] + y[5])))


def test_bf16_row_decode_layout():
    """bf16 row: w13 [2I, H] then w2 [H, I]; each entry placed by hand."""
    H, I = 4, 2
    w13 = np.arange(2 * I * H, dtype=np.float32).reshape(2 * I, H) - 3
    w2 = (np.arange(H * I, dtype=np.float32).reshape(H, I) + 1) * 0.5
    row = np.concatenate([f32_to_bf16_bits(w13).reshape(-1), f32_to_bf16_bits(w2).reshape(-1)])
    row = row.view(np.uint8)
    assert row.size == expert_row_bytes("bf16", H, I)
    a, b = expert_weights(row, "bf16", H, I)
    assert a.tolist() == w13.tolist() and b.tolist() == w2.tolist()


def test_nvfp4_row_decode_by_hand():
    """A hand-built NVFP4 row (H = I = 64): w13 row n, element kk has code
    (n + kk) % 16 and the K chunk's scale byte 0x38 + (n % 4) for its four
    16-element groups; w2 all code 0x2 (1.0) with scale 0x40 (2.0);
    global scales 0.5 and 0.25."""
    H, I = 64, 64
    o = nvfp4_offsets(H, I)
    row = np.zeros(expert_row_bytes("nvfp4", H, I), dtype=np.uint8)
    codes = np.array([[(n + kk) % 16 for kk in range(H)] for n in range(2 * I)], dtype=np.uint8)
    row[o["w13q"]:o["w13s"]] = (codes[:, 0::2] | (codes[:, 1::2] << 4)).reshape(-1)
    sc = np.zeros((H // 64, 2 * I, 4), dtype=np.uint8)
    for n in range(2 * I):
        sc[0, n, :] = 0x38 + (n % 4)
    row[o["w13s"]:o["w2q"]] = sc.reshape(-1)
    row[o["w2q"]:o["w2s"]] = 0x22
    row[o["w2s"]:o["scalars"]] = 0x40
    row[o["scalars"]:o["end"]] = np.array([0.5, 0.25, 2.0, 3.0], dtype=np.float32).view(np.uint8)
    w13, w2 = expert_weights(row, "nvfp4", H, I)
    e2m1 = [0, .5, 1, 1.5, 2, 3, 4, 6, 0, -.5, -1, -1.5, -2, -3, -4, -6]
    for n in (0, 1, 5, 127):
        s = 1.0 + (n % 4) / 8.0
        for kk in (0, 1, 15, 16, 63):
            assert w13[n, kk] == e2m1[(n + kk) % 16] * s * 0.5
    assert (w2 == 1.0 * 2.0 * 0.25).all()
    assert input_scales(row, H, I) == (2.0, 3.0)


def test_nvfp4_encoding_error_bound():
    """The generator's NVFP4 rows decode, through the oracle, to within the
    format's rounding bound of the bf16 weights they encode: |w - q| is at
    most half a grid step of the block, the step being at most 2 * sc * gs
    (between 4 and 6); with a scale layout or nibble order mix-up the error
    would be of the order of the weights themselves."""
    cfg = scaled(C1, wfmt="nvfp4", H=128, I=64, E=3)
    rows = expert_layer_rows(cfg, 0).numpy()
    bcfg = scaled(cfg, wfmt="bf16")
    brows = expert_layer_rows(bcfg, 0).numpy()     # same seed: the same bf16 weights
    for e in range(cfg.E):
        q13, q2 = expert_weights(rows[e], "nvfp4", cfg.H, cfg.I)
        b13, b2 = expert_weights(brows[e], "bf16", cfg.H, cfg.I)
        for q, b in ((q13, b13), (q2, b2)):
            blk = np.abs(b).reshape(b.shape[0], -1, 16).max(axis=-1)
            bound = np.repeat(blk / 6.0 * 1.0 + 1e-12, 16, axis=1) * (1 + 2 ** -3)
            assert (np.abs(q - b) <= bound).all()
            assert np.abs(q - b).max() < 0.2 * np.abs(b).max()
