"""Pins of the oracle's MoE FFN: a hand-worked 1-token 2-expert example, the
dense-MLP special case against a naive loop, routing invariance when every
expert is the same, and the shared-expert sum (no GPU)."""
import math

import numpy as np

import oracle
from test_oracle_codecs import _bf16_brute


def _bf16(v):
    """bf16 value nearest to v (exact rational rounding, ties to even)."""
    b = _bf16_brute(float(v))
    return float(np.array([b << 16], np.uint32).view(np.float32)[0])


def _packed(rows, cols, entries, scale=0x38, ts=1.0, block_scales=None):
    """Build packed NVFP4 with the given {(r, c): code} entries, all else code 0."""
    q = np.zeros((rows, cols), np.uint8)
    for (r, c), code in entries.items():
        q[r, c] = code
    codes = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    scales = np.full((rows, cols // 16), scale, np.uint8)
    for (r, b), s in (block_scales or {}).items():
        scales[r, b] = s
    return codes, scales, ts


def test_hand_worked_one_token_two_experts():
    H = I = 16
    x = oracle.f64_to_bf16(np.eye(1, H))           # x = e_0
    wr = np.zeros((2, H), np.float32)
    wr[1, 0] = 1.0                                   # logits (0, 1)
    experts = {
        # expert 0: g = 2 (code 4), u = 3 (code 5); down ts 2: Wd[0][0] = 1*2, Wd[1][0] = -0.5*2
        0: (_packed(I, H, {(0, 0): 4}), _packed(I, H, {(0, 0): 5}),
            _packed(H, I, {(0, 0): 2, (1, 0): 9}, ts=2.0)),
        # expert 1: g = -1 (code 10), u = 4 * 0.5 (code 6, block scale 0x30 = 0.5); Wd[2][0] = 6
        1: (_packed(I, H, {(0, 0): 10}), _packed(I, H, {(0, 0): 6}, block_scales={(0, 0): 0x30}),
            _packed(H, I, {(2, 0): 7})),
    }
    r = oracle.forward(x, wr, None, lambda e: experts[e], k=2, router_kind=oracle.ROUTER_SOFTMAX)
    assert r["ids"].tolist() == [[1, 0]]
    e1 = math.e / (1 + math.e)
    e0 = 1 / (1 + math.e)
    np.testing.assert_allclose(r["weights"][0], [e1, e0], rtol=1e-15)
    h0 = _bf16(3 * 2 / (1 + math.exp(-2)))      # W4A16: SwiGLU output rounded to bf16
    h1 = _bf16(2 * (-1) / (1 + math.exp(1)))
    want = np.zeros(H)
    want[0] = e0 * 2 * h0
    want[1] = e0 * -1 * h0
    want[2] = e1 * 6 * h1
    np.testing.assert_allclose(r["out"][0], want, rtol=1e-14, atol=1e-15)
    assert r["offsets"].tolist() == [0, 1, 2] and r["sorted_rows"].tolist() == [1, 0]


def _rand_expert(rng, H, I):
    q = lambda n, k: oracle.quantize(rng.normal(0, 0.02, (n, k)).astype(np.float32))
    return q(I, H), q(I, H), q(H, I)


def test_single_expert_is_a_dense_swiglu_mlp():
    rng = np.random.default_rng(11)
    T, H, I = 3, 32, 16
    x = oracle.f64_to_bf16(rng.normal(0, 1, (T, H)))
    ex = _rand_expert(rng, H, I)
    wr = rng.normal(0, 1, (1, H)).astype(np.float32)
    r = oracle.forward(x, wr, None, lambda e: ex, k=1, router_kind=oracle.ROUTER_SOFTMAX)
    Wg, Wu, Wd = (oracle.dequantize(*p) for p in ex)
    xs = oracle.bf16_to_f64(x)
    for t in range(T):   # naive loops
        h = []
        for i in range(I):
            g = sum(Wg[i][j] * xs[t][j] for j in range(H))
            u = sum(Wu[i][j] * xs[t][j] for j in range(H))
            h.append(_bf16(g / (1 + math.exp(-g)) * u))
        for j in range(H):
            y = sum(Wd[j][i] * h[i] for i in range(I))
            assert abs(r["out"][t][j] - y) <= 1e-12 * (1 + abs(y))


def test_identical_experts_make_routing_irrelevant():
    rng = np.random.default_rng(12)
    T, H, I, E = 9, 64, 32, 6
    x = oracle.f64_to_bf16(rng.normal(0, 1, (T, H)))
    ex = _rand_expert(rng, H, I)
    wr = rng.normal(0, 1, (E, H)).astype(np.float32)
    ref = oracle.forward(x, wr[:1], None, lambda e: ex, k=1, router_kind=oracle.ROUTER_SOFTMAX)["out"]
    for kind in (oracle.ROUTER_SOFTMAX, oracle.ROUTER_SIGMOID):
        for k in (2, 4):
            out = oracle.forward(x, wr, None, lambda e: ex, k=k, router_kind=kind)["out"]
            np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)


def test_shared_expert_adds_its_ffn():
    rng = np.random.default_rng(13)
    T, H, I, E = 5, 64, 32, 4
    x = oracle.f64_to_bf16(rng.normal(0, 1, (T, H)))
    exs = [_rand_expert(rng, H, I) for _ in range(E)]
    sh = _rand_expert(rng, H, 48)
    wr = rng.normal(0, 1, (E, H)).astype(np.float32)
    a = oracle.forward(x, wr, None, lambda e: exs[e], k=2, router_kind=oracle.ROUTER_SOFTMAX)["out"]
    b = oracle.forward(x, wr, None, lambda e: exs[e], k=2, router_kind=oracle.ROUTER_SOFTMAX, shared=sh)["out"]
    only = oracle.forward(x, wr[:1], None, lambda e: sh, k=1, router_kind=oracle.ROUTER_SOFTMAX)["out"]
    np.testing.assert_allclose(b - a, only, rtol=1e-10, atol=1e-13)


def test_w4a4_quantises_x_and_h_with_batch_tensor_scales():
    rng = np.random.default_rng(14)
    T, H, I, E = 12, 64, 32, 4
    x = oracle.f64_to_bf16(rng.normal(0, 1, (T, H)))
    exs = [_rand_expert(rng, H, I) for _ in range(E)]
    wr = rng.normal(0, 1, (E, H)).astype(np.float32)
    r4 = oracle.forward(x, wr, None, lambda e: exs[e], k=2, router_kind=oracle.ROUTER_SIGMOID,
                        mode=oracle.MODE_W4A4, keep=True)
    r16 = oracle.forward(x, wr, None, lambda e: exs[e], k=2, router_kind=oracle.ROUTER_SIGMOID)
    xc, xs, xts = oracle.quantize(oracle.bf16_to_f32(x))
    assert r4["x_ts"] == xts and np.array_equal(r4["x_codes"], xc) and np.array_equal(r4["x_scales"], xs)
    assert np.array_equal(r4["ids"], r16["ids"])
    # every h row lies on the NVFP4 grid of the batch tensor scale
    for h in r4["h"].values():
        c, s, _ = oracle.quantize(h.astype(np.float32), r4["h_ts"])
        np.testing.assert_array_equal(oracle.dequantize(c, s, r4["h_ts"]), h)
    # 4-bit activations move the output by quantisation noise only
    rel = np.linalg.norm(r4["out"] - r16["out"]) / np.linalg.norm(r16["out"])
    assert 1e-4 < rel < 0.3


def test_w4a4_hand_worked_swiglu_tensor_scales():
    """W4A4 by hand, 2 tokens, 2 routed experts (top-1) and a shared expert,
    with every value on the NVFP4 grid so each step is exact.  Pins the SwiGLU
    quantiser's tensor scale: the amax over ALL routed rows / 2688 for the
    routed experts (3528 / 2688 = 1.3125), the shared expert's own rows for its
    own scale (10584 / 2688 = 3.9375).  A per-expert amax, a routed amax that
    took in the shared rows, or another divisor each change the output."""
    H = I = 16
    x = np.zeros((2, H), np.uint16)
    x[0, 0] = x[1, 1] = int(oracle.f64_to_bf16(np.array([2688.0]))[0])   # amax 2688: x tensor scale 1
    wr = np.zeros((2, H), np.float32)
    wr[0, 0] = wr[1, 1] = 1.0                         # token 0 -> expert 0, token 1 -> expert 1
    ts_gu, ts_d = 2.0 ** -6, 2.0 ** -10
    experts = {
        # g = 2688 * 1 / 64 = 42 (silu(42) = 42 in FP64), u = 2688 * 2 / 64 = 84: h[0] = 3528
        0: (_packed(I, H, {(0, 0): 2}, ts=ts_gu), _packed(I, H, {(0, 0): 4}, ts=ts_gu),
            _packed(H, I, {(0, 0): 2, (1, 0): 9}, ts=ts_d)),          # Wd[0][0] = 1, Wd[1][0] = -0.5
        # g = 42, u = 2688 * 1.5 / 64 = 63: h[3] = 2646
        1: (_packed(I, H, {(3, 1): 2}, ts=ts_gu), _packed(I, H, {(3, 1): 3}, ts=ts_gu),
            _packed(H, I, {(2, 3): 4}, ts=ts_d)),                     # Wd[2][3] = 2
    }
    # shared: token 0 g = 63, u = 168 (h[5] = 10584); token 1 g = 42, u = 42 (h[5] = 1764)
    shared = (_packed(I, H, {(5, 0): 3, (5, 1): 2}, ts=ts_gu), _packed(I, H, {(5, 0): 6, (5, 1): 2}, ts=ts_gu),
              _packed(H, I, {(4, 5): 2}, ts=ts_d))                    # Wd[4][5] = 1
    r = oracle.forward(x, wr, None, lambda e: experts[e], k=1, router_kind=oracle.ROUTER_SOFTMAX,
                       mode=oracle.MODE_W4A4, shared=shared, keep=True)
    assert r["ids"].tolist() == [[0], [1]] and r["weights"].tolist() == [[1.0], [1.0]]
    assert r["x_ts"] == 1.0
    assert r["h_ts"] == 1.3125 and r["shared_h_ts"] == 3.9375
    # routed h, quantised with ts 1.3125:
    #   3528: s = E4M3((3528/6)/1.3125 = 448) = 448, den = 588, code 6 -> 3528
    #   2646: (2646/6)/1.3125 = 336, a tie between 320 and 352 -> 320 (even), den = 420,
    #         2646/420 = 6.3 saturates to 6 -> 6 * 320 * 1.3125 = 2520
    # shared h, ts 3.9375: 10584 -> 10584; 1764: (1764/6)/3.9375 = 74.67 -> 72, den = 283.5,
    #         1764/283.5 = 6.22 -> 6 -> 6 * 72 * 3.9375 = 1701
    assert r["h"][0][0, 0] == 3528.0 and r["h"][1][0, 3] == 2520.0
    want = np.zeros((2, H))
    want[0, 0], want[0, 1] = 3528.0 / 1024, -0.5 * 3528.0 / 1024
    want[1, 2] = 2 * 2520.0 / 1024
    want[0, 4], want[1, 4] = 10584.0 / 1024, 1701.0 / 1024
    np.testing.assert_array_equal(r["out"], want)
