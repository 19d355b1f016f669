"""Pins of the oracle's router logits, top-k, routing weights and grouping
(no GPU)."""
import itertools

import numpy as np
import pytest

import oracle


def _bf16(a):
    return oracle.f64_to_bf16(np.asarray(a, np.float64))


def test_logit_order_hand_worked():
    # Position h belongs to lane h mod 32; each lane sums in increasing h; the
    # butterfly adds lane l ^ 16, ^ 8, ^ 4, ^ 2, ^ 1.  One 2^24 term at h = 0
    # (lane 0) and two ones: where they sit decides the fp32 rounding.
    H = 256
    w = np.zeros((1, H), np.float32)
    w[0, 0] = 2.0 ** 24
    w[0, [1, 2, 3, 32]] = 1.0
    x = np.zeros((4, H))
    x[0, [0, 1, 3]] = 1.0    # lanes 1 and 3: (l1 + l3) = 2 at offset 2, then 2^24 + 2 exactly
    x[1, [0, 1, 2]] = 1.0    # lanes 1 and 2: 2^24 + l2 -> 2^24 at offset 2, + l1 -> 2^24 at offset 1
    x[2, [0, 32, 1]] = 1.0   # h = 32 is lane 0 again: (2^24 + 1) -> 2^24 inside the lane, then + l1
    x[3, [0, 3]] = 1.0       # a single one: 2^24 + 1 -> 2^24 (ties to even)
    lg = oracle.router_logits(_bf16(x), w, None)
    assert lg[0, 0] == 2.0 ** 24 + 2
    assert lg[1, 0] == 2.0 ** 24
    assert lg[2, 0] == 2.0 ** 24
    assert lg[3, 0] == 2.0 ** 24
    b = np.array([0.5], np.float32)
    assert oracle.router_logits(_bf16(x[:1]), w, b)[0, 0] == 2.0 ** 24 + 2  # bias added last in fp32


def test_logits_within_fp32_error_bound_of_exact_dot():
    rng = np.random.default_rng(6)
    T, H, E = 5, 1024, 12
    x = _bf16(rng.normal(0, 1, (T, H)))
    w = rng.normal(0, H ** -0.5, (E, H)).astype(np.float32)
    bias = rng.normal(0, 1, E).astype(np.float32)
    lg = oracle.router_logits(x, w, bias).astype(np.float64)
    xf = oracle.bf16_to_f64(x)
    exact = xf @ w.astype(np.float64).T + bias
    absdot = np.abs(xf) @ np.abs(w.astype(np.float64)).T + np.abs(bias)
    n = H // 32 + 5 + 1
    gamma = n * 2.0 ** -24 / (1 - n * 2.0 ** -24)
    assert np.all(np.abs(lg - exact) <= gamma * absdot)


def _brute_topk(lg_row, k):
    order = sorted(range(len(lg_row)), key=lambda e: (-float(lg_row[e]), e))
    return order[:k]


@pytest.mark.parametrize("E,k", [(4, 1), (6, 2), (8, 3), (5, 5)])
def test_topk_brute_force_with_ties(E, k):
    rng = np.random.default_rng(E * 10 + k)
    lg = rng.integers(-2, 3, (200, E)).astype(np.float32)  # many exact ties
    ids, w = oracle.topk(lg, k, oracle.ROUTER_SOFTMAX)
    for t in range(lg.shape[0]):
        assert list(ids[t]) == _brute_topk(lg[t], k)


def test_softmax_weights_identity_and_sum():
    rng = np.random.default_rng(7)
    lg = rng.normal(0, 2, (50, 16)).astype(np.float32)
    ids, w = oracle.topk(lg, 4, oracle.ROUTER_SOFTMAX, True)
    full = np.exp(lg.astype(np.float64))
    full /= full.sum(axis=1, keepdims=True)            # softmax over all experts
    sel = np.take_along_axis(full, ids, axis=1)
    np.testing.assert_allclose(w, sel / sel.sum(axis=1, keepdims=True), rtol=1e-12)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-12)
    ids2, w2 = oracle.topk(lg, 4, oracle.ROUTER_SOFTMAX, False)
    np.testing.assert_allclose(w2, sel, rtol=1e-12)   # no renormalisation: plain softmax probs


def test_sigmoid_weights():
    rng = np.random.default_rng(8)
    lg = rng.normal(0, 3, (50, 32)).astype(np.float32)
    ids, w = oracle.topk(lg, 8, oracle.ROUTER_SIGMOID, True)
    s = 1.0 / (1.0 + np.exp(-np.take_along_axis(lg, ids, axis=1).astype(np.float64)))
    np.testing.assert_allclose(w, s / s.sum(axis=1, keepdims=True), rtol=1e-12)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-12)
    _, w2 = oracle.topk(lg, 8, oracle.ROUTER_SIGMOID, False)
    np.testing.assert_allclose(w2, s, rtol=1e-12)


def test_group_is_a_stable_sort():
    rng = np.random.default_rng(9)
    for T, k, E in [(1, 1, 1), (7, 2, 5), (64, 8, 32), (300, 4, 7)]:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        offsets, rows = oracle.group(ids, E)
        flat = ids.ravel()
        assert np.array_equal(rows, np.argsort(flat, kind="stable"))
        assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))


def test_route_permutation_covers_every_pair_once():
    rng = np.random.default_rng(10)
    T, H, E, k = 33, 256, 9, 3
    x = _bf16(rng.normal(0, 1, (T, H)))
    w = rng.normal(0, H ** -0.5, (E, H)).astype(np.float32)
    r = oracle.route(x, w, None, k, oracle.ROUTER_SOFTMAX)
    assert sorted(r["sorted_rows"].tolist()) == list(range(T * k))
    for e in range(E):
        seg = r["sorted_rows"][r["offsets"][e]:r["offsets"][e + 1]]
        assert np.all(r["ids"].ravel()[seg] == e)
        assert np.all(np.diff(seg) > 0)


def test_bf16_router_words_widen_exactly():
    """A bf16 router weight gives the logits of its exact fp32 widening (same
    fixed order), and words off the fp32 grid of 8 bits still count in full:
    0x3F81 is 1 + 2^-7, so x = 1 at one position gives exactly that logit."""
    rng = np.random.default_rng(21)
    T, H, E = 5, 256, 7
    x = _bf16(rng.normal(0, 1, (T, H)))
    w16 = _bf16(rng.normal(0, H ** -0.5, (E, H)))
    widened = (w16.astype(np.uint32) << 16).view(np.float32)
    np.testing.assert_array_equal(oracle.router_logits(x, w16, None), oracle.router_logits(x, widened, None))
    one = np.zeros((1, H), np.uint16)
    one[0, 3] = 0x3F80                               # x = 1.0 at h = 3
    w = np.zeros((2, H), np.uint16)
    w[0, 3] = 0x3F81                                 # 1.0078125
    w[1, 3] = 0xBF00                                 # -0.5
    assert oracle.router_logits(one, w, None).tolist() == [[1.0078125, -0.5]]
