"""moe_route_static: the routing entry point that allocates nothing.

Some callers cannot call cudaMalloc at all.  Examples are code running inside
another allocator's arena or under a memory-capped runtime, and a host that
forbids device allocations after start-up.  They still need routing and
grouping.  moe_route_static keeps its scratch in a device array that lives in
the library itself.  This test calls it through the C ABI twice in a row and
checks every output against the plan-based moe_route on the same inputs."""
import ctypes

import numpy as np
import pytest
import torch

import synth
import moe_routed_expert_router_gb300 as moe
from helpers import plan_for

pytestmark = pytest.mark.gpu


def _static_route(w, x, rw, bias):
    T, k, E = x.shape[0], w.top_k, w.experts
    out = dict(topk_ids=torch.empty(T, k, dtype=torch.int32, device="cuda"),
               topk_w=torch.empty(T, k, dtype=torch.float32, device="cuda"),
               expert_offsets=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
               sorted_rows=torch.empty(max(T * k, 1), dtype=torch.int32, device="cuda"))
    st = moe.lib().moe_route_static(
        x.data_ptr(), T, w.hidden, rw.data_ptr(), None if bias is None else bias.data_ptr(), E, k,
        moe.ROUTER_SIGMOID if w.router == "sigmoid" else moe.ROUTER_SOFTMAX, int(w.renormalize),
        out["topk_ids"].data_ptr(), out["topk_w"].data_ptr(), out["expert_offsets"].data_ptr(),
        out["sorted_rows"].data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == moe.OK, moe.STATUS[st]
    torch.cuda.synchronize()
    return out


def _same(got, ref):
    # the same router and grouping kernels on the same inputs: every output,
    # the routing weights included, bit for bit
    for key in ("topk_ids", "topk_w", "expert_offsets", "sorted_rows"):
        assert torch.equal(got[key], ref[key]), key


@pytest.mark.parametrize("static_first", [False, True])
@pytest.mark.parametrize("name", ["decode4_w4a16", "prompt4096_w4a4"])
def test_static_route_matches_plan_route_twice(name, static_first):
    w = synth.WORKLOADS[name]
    with plan_for(w) as plan:
        for seed in (0, 1):   # two calls in a row through the shared array
            x = synth.activations(w, seed, device="cuda")
            rw = synth.router_weight(w, seed, "cuda")
            bias = synth.router_bias(w, seed, "cuda")
            if static_first:   # nothing the static array holds carries over into a later call
                got = _static_route(w, x, rw, bias)
            ref = plan.route(x, rw, bias)
            assert plan.sync_status() == moe.OK
            if not static_first:
                got = _static_route(w, x, rw, bias)
            _same(got, ref)


def test_static_route_after_a_plan_with_fewer_experts():
    """The routing kernels' shared-memory limits are device-wide: a plan created
    for 8 experts between two static calls for 256 experts must not lower them."""
    w = synth.WORKLOADS["prompt4096_w4a4"]
    x = synth.activations(w, 2, device="cuda")
    rw = synth.router_weight(w, 2, "cuda")
    bias = synth.router_bias(w, 2, "cuda")
    first = _static_route(w, x, rw, bias)
    small = synth.scaled(synth.WORKLOADS["tiny_w4a16"], tokens=4)
    with plan_for(small) as tiny:
        xs = synth.activations(small, 0, device="cuda")
        tiny.route(xs, synth.router_weight(small, 0, "cuda"))
        assert tiny.sync_status() == moe.OK
        again = _static_route(w, x, rw, bias)
    _same(again, first)
    with plan_for(w) as plan:
        ref = plan.route(x, rw, bias)
        assert plan.sync_status() == moe.OK
    _same(first, ref)


def test_static_route_rejects_sizes_beyond_its_array():
    L = moe.lib()
    # T * E above the array's 2^20 logits: refused before anything runs
    st = L.moe_route_static(16, 8192, 4096, 16, None, 256, 8, 0, 1, 16, 16, 16, 16, None)
    assert st == moe.ERR_UNSUPPORTED_SHAPE
