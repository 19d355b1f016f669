"""GPU quantisers against the oracle, bit for bit (codes, scales, tensor scales)."""
import numpy as np
import pytest
import torch

import oracle
import moe_routed_expert_router_gb300 as moe
from helpers import plan_for
import synth

pytestmark = pytest.mark.gpu


def _crafted(rows, cols, rng):
    x = rng.normal(0, 0.02, (rows, cols)).astype(np.float32)
    mags = np.array([0, .25, .5, .75, 1, 1.25, 1.5, 1.75, 2, 2.5, 3, 3.5, 4, 5, 6, 7], np.float32)
    x[0, :16] = mags * 0.01                     # E2M1 midpoints after scaling
    x[1, :16] = -mags * 0.01
    x[2, :16] = 0.0                             # an all-zero block
    x[2, 16:32] = -0.0
    x[3, :16] = 1e-30                           # a block far below the tensor scale
    x[4, 5] = 3.0                               # the tensor amax
    x[5, :16] = np.float32(3.0 / 6 / 448 * 6)  # exact representable scale boundary
    return x


@pytest.mark.parametrize("shape", [(1, 16), (7, 48), (64, 512), (33, 1536)])
def test_weight_quantiser_is_bit_exact(shape):
    rng = np.random.default_rng(sum(shape))
    x = _crafted(*shape, rng) if shape[0] >= 6 else rng.normal(0, 1, shape).astype(np.float32)
    q = moe.quantize_nvfp4(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    c, s, ts = oracle.quantize(x)
    assert q.ts.item() == ts
    np.testing.assert_array_equal(q.scales[0].cpu().numpy(), s)
    np.testing.assert_array_equal(q.codes[0].cpu().numpy(), c)


def test_batched_weight_quantiser_one_tensor_scale_per_item():
    rng = np.random.default_rng(3)
    x = rng.normal(0, 0.02, (5, 32, 256)).astype(np.float32)
    x[2] *= 100
    q = moe.quantize_nvfp4(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    for b in range(5):
        c, s, ts = oracle.quantize(x[b])
        assert q.ts[b].item() == ts
        np.testing.assert_array_equal(q.codes[b].cpu().numpy(), c)
        np.testing.assert_array_equal(q.scales[b].cpu().numpy(), s)


def test_all_zero_weight():
    q = moe.quantize_nvfp4(torch.zeros(4, 64, device="cuda"))
    torch.cuda.synchronize()
    assert q.ts.item() == 0.0 and not q.codes.any() and not q.scales.any()


@pytest.mark.parametrize("T,H", [(1, 256), (37, 512), (16, 7168), (4096, 7168)])
def test_activation_quantiser_is_bit_exact(T, H):
    w = synth.scaled(synth.WORKLOADS["prompt4096_w4a4"], tokens=T, hidden=H)
    x = synth.activations(w, seed=T, device="cuda")
    with plan_for(w, max_tokens=T) as plan:
        codes, scales, ts = plan.quantize_act(x)
        assert plan.sync_status() == moe.OK
    xb = x.cpu().view(torch.int16).numpy().view(np.uint16)
    c, s, t = oracle.quantize_activations(xb)
    assert ts.item() == t
    np.testing.assert_array_equal(scales.cpu().numpy(), s)
    np.testing.assert_array_equal(codes.cpu().numpy(), c)
