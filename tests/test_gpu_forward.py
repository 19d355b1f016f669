"""moe_forward against the FP64 oracle on the seeded workloads.

Tolerance on the bf16 output (the stated bar): max|d| <= 2e-2 * RMS(oracle)
and ||d||_2 / ||oracle||_2 <= 5e-3.  Routing, offsets and W4A4 activation codes
are checked bit for bit in test_gpu_route.py / test_gpu_quant.py."""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_routed_expert_router_gb300 as moe
from helpers import Case, bf16_bits, plan_for

pytestmark = pytest.mark.gpu


def _parity(case: Case, plan=None):
    out, st, plan = case.gpu_forward(plan)
    assert st == moe.OK, moe.STATUS[st]
    ref = case.oracle_forward()
    ok, stats = oracle.compare_output(bf16_bits(out), ref["out"], ref["band"])
    stats["h_flips"] = ref["h_flips"]
    assert ok, stats
    return out, ref, stats


def test_tiny_full():
    _parity(Case(synth.WORKLOADS["tiny_w4a16"], 0))


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_decode_w4a16_full(seed):
    _parity(Case(synth.WORKLOADS["decode4_w4a16"], seed))


def test_verify16_w4a4_full():
    w = synth.WORKLOADS["verify16_w4a4"]
    case = Case(w, 0)
    _parity(case)
    # another batch of the 64-batch sequence through the same plan and weights
    case.x = synth.activations(w, 0, batch=5, device="cuda")
    _parity(case)


def test_prompt512_w4a16_full():
    _parity(Case(synth.WORKLOADS["prompt512_w4a16"], 0))


@pytest.mark.parametrize("path", ["cuda_core", "tensor_core"])
def test_w4a4_paths_against_oracle(path):
    w = synth.scaled(synth.WORKLOADS["prompt4096_w4a4"], tokens=200, hidden=1024, experts=16, inter=512,
                     shared_inter=256)
    case = Case(w, 1)
    plan = plan_for(w)
    plan.set_path(moe.PATH_CUDA_CORE if path == "cuda_core" else moe.PATH_TENSOR_CORE)
    _parity(case, plan)


PATHS = {"cuda_core": moe.PATH_CUDA_CORE, "tensor_core": moe.PATH_TENSOR_CORE, "warp_mma": moe.PATH_WARP_MMA}


@pytest.mark.parametrize("path", ["cuda_core", "tensor_core", "warp_mma"])
def test_w4a16_paths_against_oracle(path):
    w = synth.scaled(synth.WORKLOADS["prompt512_w4a16"], tokens=200, hidden=1024, experts=16, inter=512,
                     shared_inter=256)
    case = Case(w, 3)
    plan = plan_for(w)
    plan.set_path(PATHS[path])
    _parity(case, plan)


@pytest.mark.parametrize("path", ["tensor_core", "warp_mma"])
@pytest.mark.parametrize("seed", [0, 1])
def test_decode_w4a16_full_on_tensor_paths(seed, path):
    w = synth.WORKLOADS["decode4_w4a16"]
    case = Case(w, seed)
    plan = plan_for(w)
    plan.set_path(PATHS[path])
    _parity(case, plan)


def test_w4a16_warp_mma_matches_cuda_core_path():
    w = synth.scaled(synth.WORKLOADS["prompt512_w4a16"], tokens=77, hidden=2048, experts=24, inter=768,
                     shared_inter=512)
    case = Case(w, 6)
    p1, p2 = plan_for(w), plan_for(w)
    p1.set_path(moe.PATH_CUDA_CORE)
    p2.set_path(moe.PATH_WARP_MMA)
    a, st1, _ = case.gpu_forward(p1)
    b, st2, _ = case.gpu_forward(p2)
    assert st1 == moe.OK and st2 == moe.OK
    d = (a.float() - b.float()).abs()
    rms = a.float().pow(2).mean().sqrt()
    assert (d.max() / rms).item() < 2e-2 and (d.norm() / a.float().norm()).item() < 5e-3


def test_w4a16_tensor_core_path_matches_cuda_core_path():
    w = synth.scaled(synth.WORKLOADS["prompt512_w4a16"], tokens=77, hidden=2048, experts=24, inter=768)
    case = Case(w, 4)
    p1, p2 = plan_for(w), plan_for(w)
    p1.set_path(moe.PATH_CUDA_CORE)
    p2.set_path(moe.PATH_TENSOR_CORE)
    a, st1, _ = case.gpu_forward(p1)
    b, st2, _ = case.gpu_forward(p2)
    assert st1 == moe.OK and st2 == moe.OK
    d = (a.float() - b.float()).abs()
    rms = a.float().pow(2).mean().sqrt()
    assert (d.max() / rms).item() < 2e-2 and (d.norm() / a.float().norm()).item() < 5e-3


def test_tensor_core_path_matches_cuda_core_path():
    w = synth.scaled(synth.WORKLOADS["verify16_w4a4"], hidden=2048, experts=32, inter=768, shared_inter=512)
    w = synth.scaled(w, inter=512)
    case = Case(w, 2)
    p1, p2 = plan_for(w), plan_for(w)
    p1.set_path(moe.PATH_CUDA_CORE)
    p2.set_path(moe.PATH_TENSOR_CORE)
    a, st1, _ = case.gpu_forward(p1)
    b, st2, _ = case.gpu_forward(p2)
    assert st1 == moe.OK and st2 == moe.OK
    d = (a.float() - b.float()).abs()
    rms = a.float().pow(2).mean().sqrt()
    assert (d.max() / rms).item() < 2e-2 and (d.norm() / a.float().norm()).item() < 5e-3


def test_prompt4096_w4a4_reduced():
    # several 128-row tiles for the heavy experts and a ragged tail
    w = synth.scaled(synth.WORKLOADS["prompt4096_w4a4"], tokens=300, hidden=1024, experts=32, inter=512)
    _parity(Case(w, 0))


@pytest.mark.parametrize("T", [1, 5, 37])
def test_ragged_token_counts(T):
    w = synth.scaled(synth.WORKLOADS["decode4_w4a16"], tokens=T, hidden=1024, experts=16, inter=256,
                     shared_inter=384)
    _parity(Case(w, T))


def test_w4a4_shared_and_sigmoid_small():
    w = synth.scaled(synth.WORKLOADS["verify16_w4a4"], tokens=9, hidden=512, experts=12, inter=256,
                     shared_inter=128)
    _parity(Case(w, 4))


def test_every_token_on_one_expert():
    w = synth.scaled(synth.WORKLOADS["tiny_w4a16"], tokens=40, top_k=1)
    case = Case(w, 3)
    case.bias = torch.full((w.experts,), -30.0, device="cuda")
    case.bias[5] = 30.0
    _, ref, _ = _parity(case)
    assert ref["offsets"][5] == 0 and ref["offsets"][6] == 40


@pytest.mark.parametrize("mode,T,path", [("w4a16", 32, "tensor_core"), ("w4a16", 33, "tensor_core"),
                                         ("w4a16", 65, "tensor_core"), ("w4a16", 16, "warp_mma"),
                                         ("w4a16", 17, "warp_mma"), ("w4a16", 33, "warp_mma"),
                                         ("w4a16", 129, "warp_mma"), ("w4a4", 128, "tensor_core"),
                                         ("w4a4", 129, "tensor_core")])
def test_tile_boundaries_on_tensor_cores(mode, T, path):
    # every token on experts 2 and 6: each holds T rows, cut into 32-row
    # (W4A16) or 128-row (W4A4) tiles with a ragged last one
    base = synth.WORKLOADS["tiny_w4a16"] if mode == "w4a16" else synth.WORKLOADS["verify16_w4a4"]
    w = synth.scaled(base, tokens=T, hidden=512, experts=8, top_k=2, inter=256, shared_inter=256)
    case = Case(w, T)
    case.bias = torch.full((w.experts,), -30.0, device="cuda")
    case.bias[2] = 30.0
    case.bias[6] = 29.0
    plan = plan_for(w)
    plan.set_path(PATHS[path])
    _, ref, _ = _parity(case, plan)
    assert ref["offsets"][3] - ref["offsets"][2] == T and ref["offsets"][7] - ref["offsets"][6] == T


def test_k_equals_e():
    w = synth.scaled(synth.WORKLOADS["tiny_w4a16"], top_k=8)
    _parity(Case(w, 5))


def test_zero_tokens_and_reuse_of_plan():
    w = synth.WORKLOADS["tiny_w4a16"]
    case = Case(w, 0)
    plan = plan_for(w)
    empty = torch.empty(0, w.hidden, dtype=torch.bfloat16, device="cuda")
    plan.forward(empty, case.rw, case.bias, case.routed, case.shared)
    assert plan.sync_status() == moe.OK
    a = _parity(case, plan)[0]
    b = _parity(case, plan)[0]          # the combine accumulator is cleared between calls
    assert torch.equal(a, b) or (a.float() - b.float()).abs().max().item() < 1e-2


def test_forward_host_matches_device_path():
    w = synth.WORKLOADS["decode4_w4a16"]
    case = Case(w, 0)
    out_dev, st, plan = case.gpu_forward()
    xh = case.x.cpu().pin_memory()
    oh = torch.empty(w.tokens, w.hidden, dtype=torch.bfloat16).pin_memory()
    plan.forward_host(xh, case.rw, case.bias, case.routed, case.shared, oh)
    assert plan.sync_status() == moe.OK
    ref = case.oracle_forward()
    ok, stats = oracle.compare_output(bf16_bits(oh), ref["out"], ref["band"])
    assert ok, stats


def test_nonfinite_refused_in_forward():
    w = synth.WORKLOADS["tiny_w4a16"]
    case = Case(w, 0)
    case.x[0, 0] = float("inf")
    _, st, _ = case.gpu_forward()
    assert st == moe.ERR_NONFINITE


def test_host_checks():
    w = synth.WORKLOADS["tiny_w4a16"]
    case = Case(w, 0)
    plan = plan_for(w)
    big = torch.zeros(w.tokens + 1, w.hidden, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        plan.forward(big, case.rw, case.bias, case.routed)
    assert e.value.status == moe.ERR_INVALID_ARG
    mis = torch.zeros(w.tokens * w.hidden + 8, dtype=torch.bfloat16, device="cuda")[1:1 + w.tokens * w.hidden]
    with pytest.raises(moe.MoeError) as e:
        plan.forward(mis.view(w.tokens, w.hidden), case.rw, case.bias, case.routed)
    assert e.value.status == moe.ERR_MISALIGNED


@pytest.mark.parametrize("name", ["decode4_w4a16", "verify16_w4a4"])
def test_forward_replays_from_a_cuda_graph(name):
    w = synth.WORKLOADS[name]
    case = Case(w, 0)
    plan = plan_for(w)
    out = torch.empty(w.tokens, w.hidden, dtype=torch.bfloat16, device="cuda")
    plan.forward(case.x, case.rw, case.bias, case.routed, case.shared, out=out)   # warm-up outside capture
    assert plan.sync_status() == moe.OK
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        plan.forward(case.x, case.rw, case.bias, case.routed, case.shared, out=out)
    out.zero_()
    for _ in range(2):
        g.replay()
    assert plan.sync_status() == moe.OK
    ref = case.oracle_forward()
    ok, stats = oracle.compare_output(bf16_bits(out), ref["out"], ref["band"])
    assert ok, stats


@pytest.mark.parametrize("name", ["decode4_w4a16", "verify16_w4a4"])
def test_forward_with_bf16_router_words(name):
    """moe_forward with the router weight in bf16 words against the oracle on
    the same words."""
    case = Case(synth.WORKLOADS[name], 1)
    case.rw = case.rw.to(torch.bfloat16)
    _parity(case)
