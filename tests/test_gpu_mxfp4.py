"""MXFP4 experts (E2M1 codes, E8M0 scales a 32-value block, no tensor scale)
on the GPU against the oracle: the device quantisers bit for bit, and
moe_forward at the stated tolerance on the engines that take MXFP4 (the
warp-level MMAs for W4A16, the tcgen05 block-scaled MMAs for W4A4, the CUDA
cores for both)."""
import numpy as np
import pytest
import torch

import oracle
import synth
import moe_routed_expert_router_gb300 as moe
from helpers import Case, bf16_bits, plan_for
from test_gpu_w4a4_stages import gpu_h_state

pytestmark = pytest.mark.gpu


def _mx(name, **kw):
    return synth.scaled(synth.WORKLOADS[name], **kw) if kw else synth.WORKLOADS[name]


@pytest.mark.parametrize("shape", [(1, 32), (7, 64), (64, 512), (33, 2048)])
def test_mx_weight_quantiser_is_bit_exact(shape):
    rng = np.random.default_rng(sum(shape) + 1)
    x = (rng.normal(0, 1, shape) * np.exp2(rng.integers(-20, 20, (shape[0], 1)))).astype(np.float32)
    if shape[0] > 5:
        x[1, :32] = 0.0                              # an all-zero block
        x[2, :32] = np.float32(2.0 ** -130)          # a subnormal amax: scale byte clamps to 0
        x[3, 0] = 8.0                                # amax on a power of two
        x[4, :4] = [7.5, 7.0, -3.0, 0.2]             # clipping above 6
    q = moe.quantize_mxfp4(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    c, s = oracle.quantize_mx(x)
    np.testing.assert_array_equal(q.scales[0].cpu().numpy(), s)
    np.testing.assert_array_equal(q.codes[0].cpu().numpy(), c)


@pytest.mark.parametrize("T,H", [(1, 512), (37, 1024), (16, 7168)])
def test_mx_activation_quantiser_is_bit_exact(T, H):
    w = synth.scaled(synth.WORKLOADS["verify16_w4a4"], tokens=T, hidden=H, inter=512, shared_inter=512)
    x = synth.activations(w, seed=T, device="cuda")
    with plan_for(w, max_tokens=T, mx=True) as plan:
        codes, scales, ts = plan.quantize_act(x)
        assert plan.sync_status() == moe.OK
    c, s = oracle.quantize_mx(oracle.bf16_to_f32(x.cpu().view(torch.int16).numpy().view(np.uint16)))
    assert ts.item() == 1.0
    np.testing.assert_array_equal(scales.cpu().numpy(), s)
    np.testing.assert_array_equal(codes.cpu().numpy(), c)


def _parity(case, plan=None):
    out, st, plan = case.gpu_forward(plan)
    assert st == moe.OK, moe.STATUS[st]
    ref = case.oracle_forward()
    ok, stats = oracle.compare_output(bf16_bits(out), ref["out"], ref["band"])
    assert ok, stats
    return out, ref


PATHS = {"auto": moe.PATH_AUTO, "cuda_core": moe.PATH_CUDA_CORE, "warp_mma": moe.PATH_WARP_MMA}


@pytest.mark.parametrize("path", ["auto", "cuda_core"])
def test_mx_decode_w4a16_full_size(path):
    """The decode workload (4 tokens, H 4096, 128 experts, I 1536, top-8, shared
    expert) with MXFP4 weights."""
    case = Case(_mx("decode4_w4a16"), 0, mx=True)
    plan = plan_for(case.w, mx=True)
    plan.set_path(PATHS[path])
    _parity(case, plan)


@pytest.mark.parametrize("path", ["warp_mma", "cuda_core"])
def test_mx_w4a16_prompt_shaped(path):
    w = _mx("prompt512_w4a16", tokens=77, hidden=2048, experts=24, inter=1024, shared_inter=512)
    case = Case(w, 5, mx=True)
    plan = plan_for(w, mx=True)
    plan.set_path(PATHS[path])
    _parity(case, plan)


@pytest.mark.parametrize("T", [1, 9, 129])
def test_mx_w4a4_on_the_cuda_cores_end_to_end_and_by_stage(T):
    w = _mx("verify16_w4a4", tokens=T, hidden=1024, experts=16, inter=512, shared_inter=512)
    case = Case(w, T, mx=True)
    plan = plan_for(w, mx=True)
    plan.set_path(moe.PATH_CUDA_CORE)
    out, st, _ = case.gpu_forward(plan)
    assert st == moe.OK, moe.STATUS[st]
    ref = case.oracle_forward()
    ok, stats = oracle.compare_output(bf16_bits(out), ref["out"], ref["band"])
    assert ok, stats
    # by stage: the GPU's own fp32 h, MXFP4-quantised by the oracle block by block
    state = gpu_h_state(plan, w, ref["offsets"], tc=False, mx=True)
    plan.close()
    for key, h in state["h"].items():
        c, s = oracle.quantize_mx(h)
        np.testing.assert_array_equal(state["codes"][key], c)
        np.testing.assert_array_equal(state["scales"][key], s)
    h_in = {e: state["h"][e] for e in state["h"]}
    ref2 = oracle.forward(case.x_host(), case.rw_host(), case.bias_host(), case.oracle_expert, k=w.top_k,
                          router_kind=oracle.ROUTER_SIGMOID, mode=oracle.MODE_W4A4,
                          shared=case.oracle_expert("shared"), h_in=h_in, fmt=oracle.FMT_MXFP4)
    ok, stats = oracle.compare_output(bf16_bits(out), ref2["out"], None)
    assert ok, stats


def _mx_stages(case, out, plan, tc):
    """The GPU's own fp32 h, MXFP4-quantised by the oracle block by block (codes
    and scales bit for bit), and the oracle's down product and combine on that h
    at the plain tolerance."""
    w = case.w
    ref = case.oracle_forward()
    state = gpu_h_state(plan, w, ref["offsets"], tc=tc, mx=True)
    for key, h in state["h"].items():
        c, s = oracle.quantize_mx(h)
        np.testing.assert_array_equal(state["scales"][key], s, err_msg=f"h scales of {key}")
        np.testing.assert_array_equal(state["codes"][key], c, err_msg=f"h codes of {key}")
    assert state["ts"] == 1.0 and state["shared_ts"] == 1.0
    ref2 = oracle.forward(case.x_host(), case.rw_host(), case.bias_host(), case.oracle_expert, k=w.top_k,
                          router_kind=oracle.ROUTER_SIGMOID, mode=oracle.MODE_W4A4,
                          shared=case.oracle_expert("shared"), h_in=dict(state["h"]), fmt=oracle.FMT_MXFP4)
    ok, stats = oracle.compare_output(bf16_bits(out), ref2["out"], None)
    assert ok, stats
    return ref


@pytest.mark.parametrize("T", [8, 64, 129])
def test_mx_w4a4_on_the_tcgen05_mmas_end_to_end_and_by_stage(T):
    """kind::mxf4 block-scaled MMAs: 8 tokens (32-row tiles), 64 (64-row
    tiles), 129 (a ragged last 128-row tile on the shared expert)."""
    w = _mx("verify16_w4a4", tokens=T, hidden=1024, experts=16, inter=512, shared_inter=1024)
    case = Case(w, T + 3, mx=True)
    plan = plan_for(w, mx=True)
    plan.set_path(moe.PATH_TENSOR_CORE)
    plan.keep_h(True)   # the gate/up launch quantises h itself; keep the fp32 h to check it
    out, st, _ = case.gpu_forward(plan)
    assert st == moe.OK, moe.STATUS[st]
    ref = _mx_stages(case, out, plan, tc=True)
    plan.close()
    ok, stats = oracle.compare_output(bf16_bits(out), ref["out"], ref["band"])
    assert ok, stats


def test_mx_w4a4_tensor_cores_quantise_h_in_the_gate_up_launch():
    """MXFP4 needs no batch amax for h, so the gate/up epilogue quantises it in
    the same pass: no separate quantiser launch, and the same codes and scales
    whether or not the fp32 h is also stored."""
    w = _mx("verify16_w4a4", tokens=64, hidden=1024, experts=16, inter=512, shared_inter=512)
    case = Case(w, 2, mx=True)
    plan = plan_for(w, mx=True)
    plan.set_path(moe.PATH_TENSOR_CORE)
    plan.set_profiling(True)
    bufs = {}
    for keep in (False, True):
        plan.keep_h(keep)
        _, st, _ = case.gpu_forward(plan)
        assert st == moe.OK, moe.STATUS[st]
        prof = plan.read_profile()
        assert prof["quant_h"][1] == 0 and prof["quant_h"][2] == 0, prof["quant_h"]
        bufs[keep] = [moe.device_view(*plan.debug_buffer(n)).clone() for n in ("h_codes", "h_scale_atoms")]
    plan.close()
    for a, b in zip(bufs[False], bufs[True]):
        assert torch.equal(a, b)


def test_mx_w4a4_full_size_verify_batch_on_the_tcgen05_mmas():
    """The 16-token verification batch at full size (H 7168, 256 experts, I
    2048, top-8, shared expert) with MXFP4 weights; AUTO takes the tcgen05 GEMMs."""
    case = Case(_mx("verify16_w4a4"), 0, mx=True)
    plan = plan_for(case.w, mx=True)
    plan.keep_h(True)
    out, st, _ = case.gpu_forward(plan)
    assert st == moe.OK, moe.STATUS[st]
    ref = _mx_stages(case, out, plan, tc=True)
    plan.close()
    ok, stats = oracle.compare_output(bf16_bits(out), ref["out"], ref["band"])
    assert ok, stats


def test_mx_plan_path_rules_and_small_shapes():
    w = _mx("verify16_w4a4", hidden=1024, experts=16, inter=512, shared_inter=512)
    with plan_for(w, mx=True) as plan:
        plan.set_path(moe.PATH_TENSOR_CORE)          # W4A4: kind::mxf4
    w16 = _mx("decode4_w4a16", hidden=1024, experts=16, inter=512, shared_inter=512)
    with plan_for(w16, mx=True) as plan:
        with pytest.raises(moe.MoeError) as e:
            plan.set_path(moe.PATH_TENSOR_CORE)      # W4A16 MXFP4: warp MMAs or CUDA cores
        assert e.value.status == moe.ERR_UNSUPPORTED_SHAPE
    with pytest.raises(moe.MoeError) as e:
        plan_for(_mx("tiny_w4a16"), mx=True)      # H 256, I 128: MXFP4 needs multiples of 512
    assert e.value.status == moe.ERR_UNSUPPORTED_SHAPE


def test_mx_scale_outside_the_f16_range_is_a_device_error_on_the_warp_mmas():
    """A weight block whose E8M0 scale lies outside 2^-23 .. 2^13 cannot be held
    exactly in the f16 operands of the warp MMAs: the kernel reports it."""
    w = _mx("decode4_w4a16", hidden=1024, experts=8, inter=512, shared_inter=512, top_k=8)
    case = Case(w, 2, mx=True)
    case.routed.gate.scales[3, 0, 0] = 60          # 2^-67 for expert 3's first gate block
    plan = plan_for(w, mx=True)
    plan.set_path(moe.PATH_WARP_MMA)
    _, st, _ = case.gpu_forward(plan)
    assert st == moe.ERR_DEVICE
