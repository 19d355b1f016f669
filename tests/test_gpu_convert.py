"""Every fp32 bit pattern through the device's fp32 -> E4M3 and fp32 -> E2M1
conversions (the ones the NVFP4 quantisers use, via moe_convert_f32) against
the oracle's scalar conversions, bit for bit.

This pins the hardware conversion (cvt.rn.satfinite) the quantisers rely on:
round to nearest even at every midpoint, saturation to the largest finite
value, subnormals, -0 and the sign of values that round to zero.  NaN inputs
are left out of the comparison: no NaN reaches a quantiser (non-finite
activations are refused, and every value a quantiser converts is a finite
ratio of finite numbers or a saturating infinity); how the two sides encode
them is reported only."""
import concurrent.futures
import os

import numpy as np
import pytest
import torch

import oracle
import moe_routed_expert_router_gb300 as moe

pytestmark = pytest.mark.gpu

CHUNK = 1 << 26
THREADS = max(1, min(16, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()))


@pytest.mark.parametrize("fmt", ["e4m3", "e2m1"])
def test_every_fp32_pattern_converts_like_the_oracle(fmt, record_property):
    host_fn = oracle.e4m3_from_f32 if fmt == "e4m3" else oracle.e2m1_from_f32
    code = moe.FMT_E4M3 if fmt == "e4m3" else moe.FMT_E2M1
    src = torch.empty(CHUNK, dtype=torch.float32).pin_memory()
    dst = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    src_d = torch.empty(CHUNK, dtype=torch.float32, device="cuda")
    nan_diff = 0
    with concurrent.futures.ThreadPoolExecutor(THREADS) as ex:
        for start in range(0, 1 << 32, CHUNK):
            bits = np.arange(start, start + CHUNK, dtype=np.uint64).astype(np.uint32)
            x = bits.view(np.float32)
            src.numpy()[:] = x
            src_d.copy_(src, non_blocking=True)
            moe.convert_f32(src_d, code, out=dst)
            want = np.concatenate(list(ex.map(host_fn, np.array_split(x, THREADS))))
            got = dst.cpu().numpy()
            nan = np.isnan(x)
            bad = (got != want) & ~nan
            if bad.any():
                i = int(np.nonzero(bad)[0][0])
                pytest.fail(f"{fmt}: fp32 0x{int(bits[i]):08x} ({x[i]!r}) -> device 0x{int(got[i]):02x}, "
                            f"oracle 0x{int(want[i]):02x}; {int(bad.sum())} mismatches in this chunk")
            nan_diff += int(((got != want) & nan).sum())
    record_property("nan_patterns_encoded_differently", nan_diff)
