"""Pins of the oracle's NVFP4 quantiser: a hand-worked golden, bounds that the
format fixes, idempotence and the tensor-scale rule (no GPU)."""
import json
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_blocks.json")


def test_hand_worked_blocks():
    g = json.load(open(GOLDEN))
    x = np.array(g["x"], np.float32).reshape(1, -1)  # four blocks in one row
    codes, scales, ts = oracle.quantize(x, g["ts"])
    assert list(scales[0]) == g["scales"]
    q = oracle.unpack_codes(codes)[0].reshape(4, 16)
    assert q.tolist() == g["codes"]
    assert list(codes[0, :8]) == g["packed_block_A"]  # low nibble = even element


def test_tensor_scale_rule():
    x = np.zeros((2, 32), np.float32)
    x[1, 5] = -2688.0
    assert oracle.tensor_scale(x) == 1.0
    codes, scales, ts = oracle.quantize(x)
    assert ts == 1.0
    assert scales[1, 0] == 0x7E  # (2688/6)/1 = 448, the largest E4M3
    assert oracle.unpack_codes(codes)[1, 5] == 0xF  # -2688 / 448 = -6
    z = np.zeros((3, 48), np.float32)
    c, s, t = oracle.quantize(z)
    assert t == 0.0 and not c.any() and not s.any()


def _e2m1_half_step(a):
    return np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0))


def test_dequantised_error_is_within_half_a_code_step():
    rng = np.random.default_rng(4)
    x = rng.normal(0, 0.02, (64, 512)).astype(np.float32)
    x[3, :16] *= 1000.0  # one block far larger than the rest
    codes, scales, ts = oracle.quantize(x)
    xh = oracle.dequantize(codes, scales, ts)
    den = np.repeat(oracle.e4m3_table()[scales], 16, axis=1) * np.float32(ts)
    v = np.abs(x.astype(np.float64)) / den
    err = np.abs(xh - x) / den
    within = v <= 6.0
    # inside the E2M1 range the error is at most half a step (plus fp32 slack)
    assert np.all(err[within] <= _e2m1_half_step(v[within]) * (1 + 1e-6) + 1e-6)
    # the block scale covers the block: amax / den <= 6 up to one E4M3 rounding (2^-4 relative)
    bamax = np.abs(x).reshape(64, -1, 16).max(axis=2)
    dec = oracle.e4m3_table()[scales] * ts
    assert np.all(bamax / dec <= 6 * (1 + 2 ** -4) + 1e-9)


def test_quantiser_is_idempotent_on_its_grid():
    rng = np.random.default_rng(5)
    x = rng.normal(0, 1, (8, 256)).astype(np.float32)
    c1, s1, t1 = oracle.quantize(x)
    xh = oracle.dequantize(c1, s1, t1).astype(np.float32)
    c2, s2, t2 = oracle.quantize(xh, t1)
    # re-quantising dequantised values with the same tensor scale keeps every code
    # whose block kept its scale
    same_scale = (s1 == s2)
    q1 = oracle.unpack_codes(c1).reshape(8, -1, 16)
    q2 = oracle.unpack_codes(c2).reshape(8, -1, 16)
    assert same_scale.mean() > 0.9
    assert np.array_equal(q1[same_scale], q2[same_scale])
