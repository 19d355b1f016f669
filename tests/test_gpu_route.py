"""moe_route against the oracle: top-k ids, expert offsets and the grouped
order bit for bit, routing weights within a few fp32 ulps (expf vs exp)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_routed_expert_router_gb300 as moe
from helpers import plan_for

pytestmark = pytest.mark.gpu


def _check(w, x, rw, bias):
    bf16 = rw.dtype == torch.bfloat16
    with plan_for(w, max_tokens=max(1, x.shape[0]), router_dtype=moe.ROUTER_BF16 if bf16 else moe.ROUTER_F32) as plan:
        r = plan.route(x, rw, bias)
        assert plan.sync_status() == moe.OK
    xb = x.cpu().view(torch.int16).numpy().view(np.uint16)
    rwh = rw.cpu().view(torch.int16).numpy().view(np.uint16) if bf16 else rw.cpu().numpy()
    ref = oracle.route(xb, rwh, None if bias is None else bias.cpu().numpy(), w.top_k,
                       oracle.ROUTER_SIGMOID if w.router == "sigmoid" else oracle.ROUTER_SOFTMAX, w.renormalize)
    np.testing.assert_array_equal(r["topk_ids"].cpu().numpy(), ref["ids"])
    np.testing.assert_array_equal(r["expert_offsets"].cpu().numpy(), ref["offsets"])
    np.testing.assert_array_equal(r["sorted_rows"].cpu().numpy()[:ref["sorted_rows"].size], ref["sorted_rows"])
    np.testing.assert_allclose(r["topk_w"].cpu().numpy(), ref["weights"], rtol=2e-6, atol=1e-7)
    return ref


@pytest.mark.parametrize("router_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_route_full_size(name, router_dtype):
    """Every workload at full size, with the router weight in fp32 and in bf16
    words (the same draw rounded to bf16): ids, offsets, order bit for bit."""
    w = synth.WORKLOADS[name]
    for seed in w.seeds[:2]:
        rw = synth.router_weight(w, seed, "cuda")
        if router_dtype == "bf16":
            rw = rw.to(torch.bfloat16)
        ref = _check(w, synth.activations(w, seed, device="cuda"), rw, synth.router_bias(w, seed, "cuda"))
        assert np.all(np.diff(ref["offsets"]) >= 0)


@pytest.mark.parametrize("T", [1, 16, 17, 300])
def test_route_bf16_router_ragged(T):
    w = synth.scaled(synth.WORKLOADS["verify16_w4a4"], tokens=T, hidden=1024, experts=96)
    _check(w, synth.activations(w, 8, device="cuda"), synth.router_weight(w, 8, "cuda").to(torch.bfloat16),
           synth.router_bias(w, 8, "cuda"))


@pytest.mark.parametrize("T", [1, 3, 37, 130])
def test_route_ragged_token_counts(T):
    w = synth.scaled(synth.WORKLOADS["prompt4096_w4a4"], tokens=T, hidden=1024, experts=64)
    _check(w, synth.activations(w, 7, device="cuda"), synth.router_weight(w, 7, "cuda"), synth.router_bias(w, 7, "cuda"))


def test_route_ties_go_to_the_lower_expert():
    w = synth.scaled(synth.WORKLOADS["tiny_w4a16"], tokens=40, experts=16, top_k=4)
    rw = synth.router_weight(w, 1, "cuda")
    rw[5] = rw[2]; rw[9] = rw[2]; rw[14] = rw[3]       # identical rows -> exactly equal logits
    ref = _check(w, synth.activations(w, 1, device="cuda"), rw, None)
    ids = ref["ids"]
    for t in range(ids.shape[0]):
        pos = {e: j for j, e in enumerate(ids[t])}
        for lo, hi in ((2, 5), (5, 9), (3, 14)):
            if lo in pos and hi in pos:
                assert pos[lo] < pos[hi]


@pytest.mark.parametrize("T", [5, 20])   # the decode-sized (fused top-k) and the tiled router
@pytest.mark.parametrize("kind,renorm", [("softmax", False), ("sigmoid", False), ("sigmoid", True)])
def test_route_normalisation_policies(kind, renorm, T):
    w = synth.scaled(synth.WORKLOADS["decode4_w4a16"], tokens=T, router=kind, renormalize=renorm)
    _check(w, synth.activations(w, 2, device="cuda"), synth.router_weight(w, 2, "cuda"), None)


def test_route_k_equals_e_and_single_expert():
    for E, k in ((8, 8), (1, 1), (1024, 32)):
        w = synth.scaled(synth.WORKLOADS["tiny_w4a16"], experts=E, top_k=k)
        _check(w, synth.activations(w, 3, device="cuda"), synth.router_weight(w, 3, "cuda"), None)


def test_nonfinite_activation_is_refused():
    w = synth.WORKLOADS["tiny_w4a16"]
    x = synth.activations(w, 0, device="cuda")
    x[3, 17] = float("nan")
    with plan_for(w) as plan:
        plan.route(x, synth.router_weight(w, 0, "cuda"))
        assert plan.sync_status() == moe.ERR_NONFINITE
        x[3, 17] = float("inf")
        plan.route(x, synth.router_weight(w, 0, "cuda"))
        assert plan.sync_status() == moe.ERR_NONFINITE
        x[3, 17] = 0.0
        plan.route(x, synth.router_weight(w, 0, "cuda"))
        assert plan.sync_status() == moe.OK


def test_bounded_wait_reports_timeout_and_context_survives():
    w = synth.WORKLOADS["tiny_w4a16"]
    with plan_for(w) as plan:
        plan.check_timeout(20_000_000)             # 20 ms bound on a barrier nobody arrives on
        assert plan.sync_status() == moe.ERR_TIMEOUT
        assert plan.sync_status() == moe.OK         # the error word was cleared
        x = synth.activations(w, 0, device="cuda")  # the context still runs work
        r = plan.route(x, synth.router_weight(w, 0, "cuda"))
        assert plan.sync_status() == moe.OK
        assert int(r["expert_offsets"][-1]) == w.tokens * w.top_k


def _padded_layout(offsets, rows, E, T, P, shared, tile_rows, pad=128):
    """The padded row layout moe_forward builds from the grouping, derived from
    the oracle's offsets and stable order: each expert's segment padded to a
    multiple of 128 rows (-1 marks a padding row), the shared expert's T token
    rows last (P + t), and the tiles of `tile_rows` rows over every segment."""
    counts = np.diff(offsets)
    seg = [-(-int(c) // pad) * pad for c in counts] + [(-(-T // pad) * pad) if shared else 0]
    poff = np.concatenate([[0], np.cumsum(seg)]).astype(np.int32)
    pad_pair = np.full(int(poff[-1]), -1, np.int32)
    tiles = []
    for e in range(E + 1):
        c = int(counts[e]) if e < E else (T if shared else 0)
        if e < E:
            pad_pair[poff[e]:poff[e] + c] = rows[offsets[e]:offsets[e] + c]
        else:
            pad_pair[poff[e]:poff[e] + c] = P + np.arange(c)
        for q in range(-(-c // tile_rows)):
            tiles.append((e, int(poff[e]) + q * tile_rows, min(tile_rows, c - q * tile_rows), 0))
    return poff, pad_pair, np.array(tiles, np.int32).reshape(-1, 4)


@pytest.mark.parametrize("mode,T,path,tile_rows", [("w4a16", 1, "warp_mma", 32), ("w4a16", 16, "warp_mma", 32),
                                                   ("w4a16", 16, "tensor_core", 64), ("w4a4", 16, "tensor_core", 128),
                                                   ("w4a4", 3, "cuda_core", 128), ("w4a4", 20, "tensor_core", 128),
                                                   ("w4a4", 300, "tensor_core", 128), ("w4a16", 300, "tensor_core", 64)])
def test_forward_grouping_matches_oracle(mode, T, path, tile_rows):
    """The grouping moe_forward runs (inside the decode router's last block for
    T <= 16, k_group up to 2048 pairs, the multi-block grouping above) against
    the oracle's grouping, bit for bit: expert offsets, the stable order, the
    padded offsets, the padded row map and the tile work list."""
    from helpers import Case
    base = synth.WORKLOADS["decode4_w4a16"] if mode == "w4a16" else synth.WORKLOADS["verify16_w4a4"]
    w = synth.scaled(base, tokens=T, hidden=512, experts=48, inter=256, shared_inter=256)
    case = Case(w, 3)
    paths = {"cuda_core": moe.PATH_CUDA_CORE, "tensor_core": moe.PATH_TENSOR_CORE, "warp_mma": moe.PATH_WARP_MMA}
    with plan_for(w) as plan:
        plan.set_path(paths[path])
        for _ in range(2):   # the second call must not depend on what the first one left behind
            _, st, _ = case.gpu_forward(plan)
            assert st == moe.OK
        bufs = {n: moe.device_view(*plan.debug_buffer(n)).view(torch.int32).cpu().numpy()
                for n in ("offsets", "sorted", "padded_offsets", "pad_pair", "tiles")}
    ref = oracle.route(case.x_host(), case.rw_host(), case.bias_host(), w.top_k,
                       oracle.ROUTER_SIGMOID if w.router == "sigmoid" else oracle.ROUTER_SOFTMAX, w.renormalize)
    E, P = w.experts, T * w.top_k
    poff, pad_pair, tiles = _padded_layout(ref["offsets"], ref["sorted_rows"], E, T, P, True, tile_rows)
    np.testing.assert_array_equal(bufs["offsets"][:E + 1], ref["offsets"])
    np.testing.assert_array_equal(bufs["sorted"][:P], ref["sorted_rows"])
    np.testing.assert_array_equal(bufs["padded_offsets"][:E + 2], poff)
    np.testing.assert_array_equal(bufs["pad_pair"][:poff[-1]], pad_pair)
    np.testing.assert_array_equal(bufs["tiles"].reshape(-1, 4)[:len(tiles)], tiles)


@pytest.mark.parametrize("T,E", [(256, 64), (257, 64), (300, 1024)])
def test_route_grouping_around_the_multi_block_switch(T, E):
    """Batches of up to 2048 (token, slot) pairs group in one block, larger ones
    over blocks of 1024 pairs (per-block counts, scan, placement): both sides of
    the switch, and the largest expert count (the placement's biggest shared
    memory), against the oracle bit for bit."""
    w = synth.scaled(synth.WORKLOADS["prompt4096_w4a4"], tokens=T, hidden=512, experts=E, top_k=8)
    _check(w, synth.activations(w, 11, device="cuda"), synth.router_weight(w, 11, "cuda"), synth.router_bias(w, 11, "cuda"))


def test_coexisting_plans_with_different_expert_counts():
    """Two live plans, 256 and 8 experts: the one created first still groups
    (one-block grouping, whose shared memory grows with the expert count) after
    the second exists, and both match the oracle."""
    big = synth.scaled(synth.WORKLOADS["prompt4096_w4a4"], tokens=200, hidden=512)
    small = synth.scaled(synth.WORKLOADS["tiny_w4a16"], tokens=40)
    xb, rb, bb = synth.activations(big, 5, device="cuda"), synth.router_weight(big, 5, "cuda"), \
        synth.router_bias(big, 5, "cuda")
    xs, rs = synth.activations(small, 5, device="cuda"), synth.router_weight(small, 5, "cuda")
    with plan_for(big) as p_big, plan_for(small) as p_small:
        for _ in range(2):
            got_b = p_big.route(xb, rb, bb)
            assert p_big.sync_status() == moe.OK
            got_s = p_small.route(xs, rs)
            assert p_small.sync_status() == moe.OK
        for w, x, rw, bias, got in ((big, xb, rb, bb, got_b), (small, xs, rs, None, got_s)):
            ref = oracle.route(x.cpu().view(torch.int16).numpy().view(np.uint16), rw.cpu().numpy(),
                               None if bias is None else bias.cpu().numpy(), w.top_k,
                               oracle.ROUTER_SIGMOID if w.router == "sigmoid" else oracle.ROUTER_SOFTMAX,
                               w.renormalize)
            np.testing.assert_array_equal(got["topk_ids"].cpu().numpy(), ref["ids"])
            np.testing.assert_array_equal(got["expert_offsets"].cpu().numpy(), ref["offsets"])
            np.testing.assert_array_equal(got["sorted_rows"].cpu().numpy()[:ref["sorted_rows"].size],
                                          ref["sorted_rows"])
