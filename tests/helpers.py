"""Shared set-up for the GPU parity tests: inputs are drawn once with `synth`
(on the GPU, or the CPU for small tensors), the CUDA path quantises its own
weights with moe_quantize_nvfp4 and the oracle quantises the same fp32 bytes
with its own quantiser."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
import synth
import moe_routed_expert_router_gb300 as moe

PROJ = ("gate", "up", "down")


def plan_for(w: synth.Workload, max_tokens=None, router_dtype=moe.ROUTER_F32, mx=False) -> moe.Plan:
    return moe.Plan(w.hidden, w.inter, w.experts, w.top_k, max_tokens or w.tokens,
                    router=moe.ROUTER_SIGMOID if w.router == "sigmoid" else moe.ROUTER_SOFTMAX,
                    renormalize=w.renormalize, mode=moe.W4A4 if w.mode == "w4a4" else moe.W4A16,
                    has_shared=w.shared_inter > 0, shared_inter=w.shared_inter, router_dtype=router_dtype,
                    weight_format=moe.WEIGHTS_MXFP4 if mx else moe.WEIGHTS_NVFP4)


class Case:
    """One seeded problem instance: device tensors for the CUDA path and a lazy
    per-expert oracle view of the same weights."""

    def __init__(self, w: synth.Workload, seed: int = 0, batch: int = 0, device="cuda", mx=False):
        self.w, self.seed, self.device, self.mx = w, seed, device, mx
        self.x = synth.activations(w, seed, batch, device=device)
        self.rw = synth.router_weight(w, seed, device=device)
        self.bias = synth.router_bias(w, seed, device=device)
        E, I, H = w.experts, w.inter, w.hidden
        self.routed = moe.ExpertSet(*[self._alloc(E, *self._shape(p, I)) for p in PROJ])
        for e in range(E):
            for p, t in zip(PROJ, (self.routed.gate, self.routed.up, self.routed.down)):
                wf = synth.expert_weight(w, seed, e, p, device=device)
                if mx:
                    moe.quantize_mxfp4(wf, out=moe.NvfpTensor(t.codes[e:e + 1], t.scales[e:e + 1], None))
                else:
                    moe.quantize_nvfp4(wf, out=moe.NvfpTensor(t.codes[e:e + 1], t.scales[e:e + 1], t.ts[e:e + 1]))
        self.shared = None
        if w.shared_inter:
            q = moe.quantize_mxfp4 if mx else moe.quantize_nvfp4
            self.shared = moe.ExpertSet(*[q(synth.expert_weight(w, seed, "shared", p, device)) for p in PROJ])
        torch.cuda.synchronize()

    def _shape(self, p, I):
        H = self.w.hidden
        return (I, H) if p in ("gate", "up") else (H, I)

    def _alloc(self, n, rows, cols):
        d = self.device
        return moe.NvfpTensor(torch.empty(n, rows, cols // 2, dtype=torch.uint8, device=d),
                              torch.empty(n, rows, cols // (32 if self.mx else 16), dtype=torch.uint8, device=d),
                              None if self.mx else torch.empty(n, dtype=torch.float32, device=d))

    # ---- oracle side (host copies of the same inputs, oracle quantisation)
    def x_host(self):
        return self.x.cpu().view(torch.int16).numpy().view(np.uint16)

    def rw_host(self):
        """The router weight as the oracle takes it: fp32, or bf16 words (uint16)."""
        if self.rw.dtype == torch.bfloat16:
            return self.rw.cpu().view(torch.int16).numpy().view(np.uint16)
        return self.rw.cpu().numpy()

    def bias_host(self):
        return None if self.bias is None else self.bias.cpu().numpy()

    @functools.lru_cache(maxsize=None)
    def oracle_expert(self, e):
        q = (lambda a: oracle.quantize_mx(a) + (None,)) if self.mx else oracle.quantize
        return tuple(q(synth.expert_weight(self.w, self.seed, e, p, device=self.device).cpu().numpy()) for p in PROJ)

    def oracle_forward(self, keep=False):
        w = self.w
        return oracle.forward(self.x_host(), self.rw_host(), self.bias_host(), self.oracle_expert,
                              k=w.top_k, router_kind=oracle.ROUTER_SIGMOID if w.router == "sigmoid" else
                              oracle.ROUTER_SOFTMAX, renormalize=w.renormalize,
                              mode=oracle.MODE_W4A4 if w.mode == "w4a4" else oracle.MODE_W4A16,
                              shared=self.oracle_expert("shared") if w.shared_inter else None, keep=keep,
                              fmt=oracle.FMT_MXFP4 if self.mx else oracle.FMT_NVFP4)

    def gpu_forward(self, plan=None):
        plan = plan or plan_for(self.w, router_dtype=moe.ROUTER_BF16 if self.rw.dtype == torch.bfloat16
                                else moe.ROUTER_F32, mx=self.mx)
        out = plan.forward(self.x, self.rw, self.bias, self.routed, self.shared)
        st = plan.sync_status()
        return out, st, plan


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)
