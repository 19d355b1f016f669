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


# ---- the W4A4 flip band (near-boundary quantiser decisions)

def test_flip_band_is_empty_far_from_boundaries():
    # every value exactly on an E2M1 point of a power-of-two scale; the scale
    # argument (bamax/6)/ts = 2 is itself an E4M3 value
    ts = 1.0
    x = np.array([[6.0, -4.0, 3.0, 2.0, 1.5, 1.0, 0.5, 0.0, -6.0, 4.0, -3.0, 2.0, -1.5, 1.0, -0.5, 0.0]]) * 2.0
    deq, flip, n = oracle.quant_decisions(x.astype(np.float32), ts)
    assert n == 0 and not flip.any()
    np.testing.assert_array_equal(deq, x)


def test_flip_band_of_a_code_on_a_midpoint():
    # scale 2 (as above); one value at 2.5 * den, halfway between codes 2 and 3
    x = np.array([[12.0] + [1.0] * 14 + [5.0]], np.float32)    # 5.0 / 2 = 2.5
    deq, flip, n = oracle.quant_decisions(x, 1.0)
    assert n == 1
    assert deq[0, 15] == 4.0                  # RNE: 2.5 -> 2 (even), times den 2
    np.testing.assert_array_equal(flip[0, :15], 0.0)
    assert flip[0, 15] == 2.0                 # the other side: code 3, one step (1.0) x den 2


def test_flip_band_of_a_scale_on_a_midpoint():
    # (bamax/6)/ts = 12.75/6 = 2.125, halfway between E4M3 2.0 and 2.25: RNE
    # keeps 2.0; the band is the block re-quantised with 2.25
    x = np.array([[12.75, 3.0, -1.0, 7.0] + [0.0] * 12], np.float32)
    deq, flip, n = oracle.quant_decisions(x, 1.0)
    assert n >= 1
    nom = oracle.dequantize(*oracle.quantize(x, 1.0)[:2], 1.0)
    np.testing.assert_array_equal(deq, nom)
    alt = oracle.e2m1_table()[oracle.e2m1_from_f32(x / np.float32(2.25))] * 2.25
    assert np.all(flip[0] >= np.abs(alt - nom[0]) - 1e-12)
    assert np.any(flip[0] > 0)                # the elements that move carry the band


def test_flip_band_covers_every_flip_of_small_perturbations():
    rng = np.random.default_rng(21)
    x = (rng.standard_normal((256, 1024)) * rng.uniform(0.01, 3.0, (256, 1))).astype(np.float32)
    ts = float(np.float32(oracle.tensor_scale(x) * 1.37))
    deq, flip, n = oracle.quant_decisions(x, ts)
    moved = np.zeros_like(deq)
    # perturbations 4x inside the band's margin (2^-16)
    for dx, dts in ((2.0 ** -18, 0.0), (-2.0 ** -18, 0.0), (0.0, 2.0 ** -18), (0.0, -2.0 ** -18)):
        x2 = (x.astype(np.float64) * (1 + dx)).astype(np.float32)
        t2 = float(np.float32(ts * (1 + dts)))
        d2 = oracle.dequantize(*oracle.quantize(x2, t2)[:2], t2)
        # compare at the nominal scale: changes of the decisions, not of ts itself
        moved = np.maximum(moved, np.abs(d2 * (ts / t2) - deq))
    changed = moved > 1e-6 * np.abs(deq).max()
    assert changed.sum() >= 5, "the perturbations should flip a few decisions in 256K values"
    assert np.all(flip[changed] >= moved[changed] * (1 - 1e-12))
    assert n < 0.01 * x.size                 # few decisions sit that close to a boundary


def test_bf16_half_ulp_and_output_tolerance():
    """Half a bf16 ulp: 2^(e-8) in [2^e, 2^(e+1)).  The output check lets an
    exactly rounded bf16 output pass even where its rounding alone exceeds
    2e-2 * RMS, and still fails an output two ulps away."""
    assert oracle.bf16_half_ulp(np.array([1.0, 1.99, 4.0, 6.5, -0.75, 0.0])).tolist() == \
        [2 ** -8, 2 ** -8, 2 ** -6, 2 ** -6, 2 ** -9, 2 ** -134]
    rng = np.random.default_rng(7)
    ref = rng.normal(0, 0.7, 4096)
    ref[5] = 4.0 + 0.999 * 2 ** -5 / 2            # just below the midpoint of 4 and 4 + 2^-5
    exact = oracle.f64_to_bf16(ref)               # the exactly rounded output
    rms = np.sqrt(np.mean(ref ** 2))
    assert abs(oracle.bf16_to_f64(exact[5:6])[0] - ref[5]) > 2e-2 * rms   # rounding alone exceeds the plain bar
    ok, st = oracle.compare_output(exact, ref)
    assert ok, st
    worse = exact.copy()
    worse[5] += 2                                  # two bf16 ulps up: 4.0625
    assert not oracle.compare_output(worse, ref)[0]
