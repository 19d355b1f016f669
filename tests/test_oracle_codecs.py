"""Pins of the oracle's E2M1 / E4M3 / bf16 codecs against fixed tables,
library conversions and brute force (no GPU)."""
import fractions
import math

import numpy as np
import pytest
import torch

import oracle


def test_e2m1_table_matches_spec():
    # OCP Microscaling E2M1 magnitudes; code bit 3 is the sign.
    spec = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    t = oracle.e2m1_table()
    assert list(t[:8]) == spec
    assert list(t[8:]) == [-v for v in spec]
    assert math.copysign(1.0, t[8]) == -1.0  # code 8 is -0


def test_e4m3_table_matches_torch_float8():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    t = oracle.e4m3_table()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(t), nan)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(t[~nan], ref[~nan])
    assert t[0x7E] == 448.0 and t[0x01] == 2.0 ** -9 and t[0x38] == 1.0


def _e4m3_all_finite_positive():
    t = oracle.e4m3_table()
    return np.array([t[c] for c in range(0x7F)])


def test_e4m3_quantiser_matches_torch_on_grid_midpoints_and_random():
    vals = _e4m3_all_finite_positive()
    mids = (vals[:-1] + vals[1:]) / 2  # exact in fp32 (few significant bits)
    rng = np.random.default_rng(1)
    rnd = np.concatenate([
        rng.uniform(0, 448, 20000), 2.0 ** rng.uniform(-12, 8.8, 20000), rng.uniform(0, 2 ** -6, 5000)])
    x = np.concatenate([vals, mids, rnd]).astype(np.float32)
    x = x[x <= 448]
    x = np.concatenate([x, -x])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_from_f32(x)
    assert np.array_equal(got, ref)


def test_e4m3_quantiser_saturates():
    x = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e9, np.float32(3.4e38)], np.float32)
    assert list(oracle.e4m3_from_f32(x)) == [0x7E] * len(x)
    assert list(oracle.e4m3_from_f32(-x)) == [0xFE] * len(x)


def _nearest_even(v, table_mag):
    """Brute force: nearest magnitude in the table, ties to the even code."""
    a = abs(fractions.Fraction(v))
    best = None
    for c, m in enumerate(table_mag):
        d = abs(a - fractions.Fraction(m))
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1]


def test_e2m1_quantiser_hand_midpoints():
    cases = {0.0: 0, 0.25: 0, 0.2500001: 1, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6,
             5.0001: 7, 6.0: 7, 7.0: 7, 1e30: 7, 0.5: 1, 3.0: 5, 2.9: 5, 4.5: 6}
    for v, c in cases.items():
        assert oracle.e2m1_from_f32([v])[0] == c, v
        assert oracle.e2m1_from_f32([-v])[0] == (c | 8), -v
    assert oracle.e2m1_from_f32([-0.1])[0] == 8  # a negative value keeps its sign at zero


def test_e2m1_quantiser_brute_force():
    mags = oracle.e2m1_table()[:8]
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.uniform(-7, 7, 3000), (mags[:-1] + mags[1:]) / 2,
                        -(mags[:-1] + mags[1:]) / 2]).astype(np.float32)
    got = oracle.e2m1_from_f32(x)
    for v, g in zip(x, got):
        v = float(v)
        want = 7 if abs(v) >= 6 else _nearest_even(v, mags)
        if math.copysign(1.0, v) < 0:
            want |= 8
        assert g == want, (v, g, want)


def test_round_trip_every_finite_code():
    t2 = oracle.e2m1_table()
    assert list(oracle.e2m1_from_f32(t2.astype(np.float32))) == list(range(16))
    t4 = oracle.e4m3_table()
    finite = [c for c in range(256) if not np.isnan(t4[c])]
    assert list(oracle.e4m3_from_f32(t4[finite].astype(np.float32))) == finite


def _bf16_brute(d):
    """Nearest bf16 to the double d by exact rational comparison, ties to even."""
    if d == 0:
        return 0x8000 if math.copysign(1, d) < 0 else 0
    a = fractions.Fraction(abs(d))
    e = math.floor(math.log2(abs(d)))
    while fractions.Fraction(2) ** e > a:
        e -= 1
    while fractions.Fraction(2) ** (e + 1) <= a:
        e += 1
    step = fractions.Fraction(2) ** (max(e, -126) - 7)
    lo = (a // step) * step
    hi = lo + step
    pick = lo if (a - lo < hi - a or (a - lo == hi - a and (lo / step) % 2 == 0)) else hi
    f = np.float32(float(pick))
    bits = int(np.array([f]).view(np.uint32)[0]) >> 16
    return bits | (0x8000 if d < 0 else 0)


def test_f64_to_bf16_brute_force_and_torch():
    rng = np.random.default_rng(3)
    d = np.concatenate([rng.normal(0, 1, 2000), rng.normal(0, 1e-38, 200), 2.0 ** rng.uniform(-130, 120, 500)])
    # values sitting on bf16 midpoints plus a tiny FP64 excess: a path through fp32 would round twice
    base = rng.normal(0, 1, 200).astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
    mid = (base | np.uint32(0x8000)).view(np.float32).astype(np.float64)
    d = np.concatenate([d, mid, mid * (1 + 2.0 ** -40), mid * (1 - 2.0 ** -40)])
    got = oracle.f64_to_bf16(d)
    for v, g in zip(d, got):
        assert g == _bf16_brute(float(v)), v
    f = rng.normal(0, 3, 5000).astype(np.float32)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.f64_to_bf16(f.astype(np.float64)), ref)
