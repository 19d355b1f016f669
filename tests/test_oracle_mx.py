"""Pins of the oracle's MXFP4 codec and quantiser (no GPU): the full E8M0
table against torch's float8_e8m0fnu, hand-worked blocks, the OCP MX rule
against a brute-force restatement on random blocks, the error bound, and the
FFN with MXFP4 weights against a naive loop."""
import fractions
import json
import math
import os

import numpy as np
import torch

import oracle
from test_oracle_codecs import _nearest_even
from test_oracle_ffn import _bf16

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mxfp4_blocks.json")


def test_e8m0_table_matches_torch():
    t = oracle.e8m0_table()
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    assert np.isnan(t[255]) and np.isnan(ref[255])
    np.testing.assert_array_equal(t[:255], ref[:255])
    assert t[127] == 1.0 and t[0] == 2.0 ** -127 and t[254] == 2.0 ** 127


def test_hand_worked_blocks():
    g = json.load(open(GOLDEN))
    x = np.array(g["x"], np.float32).reshape(1, -1)
    codes, scales = oracle.quantize_mx(x)
    assert list(scales[0]) == g["scales"]
    assert oracle.unpack_codes(codes)[0].reshape(-1, 32).tolist() == g["codes"]
    assert list(codes[0, :8]) == g["packed_block_A"]


def _brute_block(v):
    """The OCP MX conversion of one block, restated with exact rationals."""
    v = [float(a) for a in v]
    amax = max(abs(a) for a in v)
    if amax == 0:
        return 0, [0] * 32
    e = math.frexp(amax)[1] - 1 - 2
    s = min(max(e + 127, 0), 254)
    X = fractions.Fraction(2) ** (s - 127)
    mags = oracle.e2m1_table()[:8]
    out = []
    for a in v:
        r = fractions.Fraction(a) / X
        c = 7 if abs(r) >= 6 else _nearest_even(float(r), mags)
        if math.copysign(1.0, a) < 0:
            c |= 8
        out.append(c)
    return s, out


def test_quantiser_matches_the_rule_on_random_blocks():
    rng = np.random.default_rng(31)
    x = (rng.normal(0, 1, (40, 64)) * np.exp2(rng.integers(-30, 30, (40, 1)))).astype(np.float32)
    x[3, :32] = 0.0
    x[5, 7] = -x[5, 7]
    codes, scales = oracle.quantize_mx(x)
    q = oracle.unpack_codes(codes)
    for r in range(40):
        for b in range(2):
            s, c = _brute_block(x[r, 32 * b:32 * b + 32])
            assert scales[r, b] == s, (r, b)
            assert q[r, 32 * b:32 * b + 32].tolist() == c, (r, b)


def test_error_bound_and_clipping():
    rng = np.random.default_rng(32)
    x = rng.normal(0, 0.02, (64, 256)).astype(np.float32)
    codes, scales = oracle.quantize_mx(x)
    xh = oracle.dequantize_mx(codes, scales)
    X = np.repeat(oracle.e8m0_table()[scales], 32, axis=1)
    v = np.abs(x.astype(np.float64)) / X
    half = np.where(v < 2, 0.25, np.where(v < 4, 0.5, 1.0))
    inside = v <= 6
    assert np.all(np.abs(xh - x)[inside] / X[inside] <= half[inside] * (1 + 1e-9))
    # amax / scale lies in [4, 8): values above 6 are clipped to 6 (by at most 2 scale units)
    bm = np.abs(x).reshape(64, -1, 32).max(axis=2) / oracle.e8m0_table()[scales]
    assert np.all((bm >= 4) & (bm < 8))
    assert np.all(np.abs(xh - x)[~inside] / X[~inside] <= 2.0)


def test_quantiser_is_idempotent_on_its_grid():
    rng = np.random.default_rng(33)
    x = rng.normal(0, 1, (8, 128)).astype(np.float32)
    c, s = oracle.quantize_mx(x)
    xh = oracle.dequantize_mx(c, s).astype(np.float32)
    c2, s2 = oracle.quantize_mx(xh)
    assert np.array_equal(c, c2) and np.array_equal(s, s2)


def _mx_expert(rng, H, I):
    q = lambda n, k: oracle.quantize_mx(rng.normal(0, 0.02, (n, k)).astype(np.float32)) + (None,)
    return q(I, H), q(I, H), q(H, I)


def test_single_mx_expert_is_a_dense_swiglu_mlp():
    rng = np.random.default_rng(34)
    T, H, I = 3, 64, 32
    x = oracle.f64_to_bf16(rng.normal(0, 1, (T, H)))
    ex = _mx_expert(rng, H, I)
    wr = rng.normal(0, 1, (1, H)).astype(np.float32)
    r = oracle.forward(x, wr, None, lambda e: ex, k=1, router_kind=oracle.ROUTER_SOFTMAX, fmt=oracle.FMT_MXFP4)
    Wg, Wu, Wd = (oracle.dequantize_mx(p[0], p[1]) for p in ex)
    xs = oracle.bf16_to_f64(x)
    for t in range(T):
        h = []
        for i in range(I):
            g = sum(Wg[i][j] * xs[t][j] for j in range(H))
            u = sum(Wu[i][j] * xs[t][j] for j in range(H))
            h.append(_bf16(g / (1 + math.exp(-g)) * u))
        for j in range(H):
            y = sum(Wd[j][i] * h[i] for i in range(I))
            assert abs(r["out"][t][j] - y) <= 1e-12 * (1 + abs(y))


def test_w4a4_mx_quantises_x_and_h_block_by_block():
    rng = np.random.default_rng(35)
    T, H, I, E = 12, 64, 32, 4
    x = oracle.f64_to_bf16(rng.normal(0, 1, (T, H)))
    exs = [_mx_expert(rng, H, I) for _ in range(E)]
    wr = rng.normal(0, 1, (E, H)).astype(np.float32)
    r4 = oracle.forward(x, wr, None, lambda e: exs[e], k=2, router_kind=oracle.ROUTER_SIGMOID,
                        mode=oracle.MODE_W4A4, keep=True, fmt=oracle.FMT_MXFP4)
    r16 = oracle.forward(x, wr, None, lambda e: exs[e], k=2, router_kind=oracle.ROUTER_SIGMOID,
                         fmt=oracle.FMT_MXFP4)
    xc, xs = oracle.quantize_mx(oracle.bf16_to_f32(x))
    assert np.array_equal(r4["x_codes"], xc) and np.array_equal(r4["x_scales"], xs) and r4["x_ts"] == 1.0
    for h in r4["h"].values():   # every h row lies on its own MXFP4 grid (no batch tensor scale)
        c, s = oracle.quantize_mx(h.astype(np.float32))
        np.testing.assert_array_equal(oracle.dequantize_mx(c, s), h)
    rel = np.linalg.norm(r4["out"] - r16["out"]) / np.linalg.norm(r16["out"])
    assert 1e-4 < rel < 0.3


def test_mx_flip_band_covers_every_flip_of_small_perturbations():
    rng = np.random.default_rng(36)
    x = rng.normal(0, 1, (16, 256)).astype(np.float32)
    x[2, 0] = 4.0                     # block amax on a power of two
    x[3, 5] = np.float32(2.5 * 2 ** -1)   # a code on a midpoint (scale 2^-1 if 5.x is the block amax)
    deq, flip, n = oracle.mx_quant_decisions(x, margin=2.0 ** -16)
    assert n > 0
    for sgn in (1, -1):
        y = (x.astype(np.float64) * (1 + sgn * 2.0 ** -18)).astype(np.float32)
        c, s = oracle.quantize_mx(y)
        d = np.abs(oracle.dequantize_mx(c, s) - deq)
        assert np.all(d <= flip + 1e-12 * np.abs(deq) + 1e-30)
