"""Seeded synthetic inputs for the routed MoE FFN workloads.

This module holds no arithmetic of the method (no quantisation, routing or
FFN): it only draws random numbers.  Both the CUDA path and the CPU oracle take
their inputs from here; a test draws every tensor once, on one device, and hands
copies of the same bytes to both sides.

Recipe (the pages' workloads, stood in for by seeded synthetic data):
  * activations x ~ N(0, 1), rounded to bf16;
  * router weight Wr ~ N(0, 1/sqrt(H)) in fp32 (second argument = std);
  * expert gate/up/down weights ~ N(0, 0.02) in fp32; each side quantises them
    to NVFP4 itself (tensor scale amax/(6*448), E4M3 block scales, RNE codes);
  * a Zipf(s=1.1) router bias over a seeded expert permutation where the
    workload asks for it: bias[e] = ln p(rank(e)), p(r) = r^-1.1 / sum_q q^-1.1,
    so the softmax of the bias alone is the Zipf law.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    tokens: int            # T
    hidden: int            # H
    experts: int           # E
    inter: int             # I, per-expert intermediate
    top_k: int
    mode: str              # "w4a16" | "w4a4"
    router: str            # "softmax" | "sigmoid"
    renormalize: bool = True
    shared_inter: int = 0  # 0 = no shared expert
    zipf: bool = False
    batches: int = 1       # activation batches in one measured sequence
    seeds: tuple = (0,)
    description: str = ""

    @property
    def pairs(self) -> int:
        return self.tokens * self.top_k


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_w4a16", 16, 256, 8, 128, 2, "w4a16", "softmax",
                 description="16 tokens, H 256, 8 experts, I 128, top-2, softmax, W4A16"),
        Workload("decode4_w4a16", 4, 4096, 128, 1536, 8, "w4a16", "softmax", shared_inter=1536,
                 seeds=tuple(range(10)),
                 description="decode: 4 tokens, H 4096, 128 experts, I 1536, top-8, shared expert, W4A16"),
        Workload("prompt512_w4a16", 512, 4096, 128, 1536, 8, "w4a16", "softmax", zipf=True,
                 description="prompt: 512 tokens, H 4096, 128 experts, I 1536, top-8, Zipf bias, W4A16"),
        Workload("prompt4096_w4a4", 4096, 7168, 256, 2048, 8, "w4a4", "sigmoid", zipf=True,
                 description="long prompt: 4096 tokens, H 7168, 256 experts, I 2048, top-8, sigmoid, Zipf, W4A4"),
        Workload("verify16_w4a4", 16, 7168, 256, 2048, 8, "w4a4", "sigmoid", shared_inter=2048, zipf=True,
                 batches=64,
                 description="draft verify: 4 requests x 4 rows, H 7168, 256 experts, I 2048, top-8, shared, "
                             "Zipf, W4A4, 64 batches"),
    ]
}


def scaled(w: Workload, **kw) -> Workload:
    """A smaller (or otherwise changed) copy of a workload, for parity tests."""
    d = dataclasses.asdict(w)
    d.update(kw)
    return Workload(**d)


def _seed_of(*keys) -> int:
    h = hashlib.sha256(repr(keys).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, *keys) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(_seed_of(*keys))
    return g


def activations(w: Workload, seed: int, batch: int = 0, device="cpu") -> torch.Tensor:
    """x ~ N(0,1) as bf16 [T][H], drawn on the CPU (small), then moved."""
    g = _gen("cpu", "x", w.tokens, w.hidden, seed, batch)
    x = torch.randn(w.tokens, w.hidden, generator=g, dtype=torch.float32)
    return x.to(torch.bfloat16).to(device)


def router_weight(w: Workload, seed: int, device="cpu") -> torch.Tensor:
    """Wr ~ N(0, 1/sqrt(H)) in fp32 [E][H]."""
    g = _gen("cpu", "router", w.experts, w.hidden, seed)
    r = torch.randn(w.experts, w.hidden, generator=g, dtype=torch.float32) * (1.0 / math.sqrt(w.hidden))
    return r.to(device)


def router_bias(w: Workload, seed: int, device="cpu"):
    """Zipf(1.1) log-prior over a seeded permutation of the experts, or None."""
    if not w.zipf:
        return None
    g = _gen("cpu", "zipf", w.experts, seed)
    perm = torch.randperm(w.experts, generator=g).numpy()
    ranks = np.arange(1, w.experts + 1, dtype=np.float64)
    p = ranks ** -1.1
    p /= p.sum()
    bias = np.log(p)[perm].astype(np.float32)
    return torch.from_numpy(bias).to(device)


def expert_weight(w: Workload, seed: int, expert, proj: str, device="cpu") -> torch.Tensor:
    """One expert projection ~ N(0, 0.02) in fp32.

    expert: an index in [0, E) or "shared".  proj: "gate" | "up" ([I][H]) or
    "down" ([H][I]).  Drawn on `device`; the same (seed, expert, proj, device)
    always gives the same bytes.
    """
    inter = w.shared_inter if expert == "shared" else w.inter
    shape = (inter, w.hidden) if proj in ("gate", "up") else (w.hidden, inter)
    g = _gen(device, "expert", w.hidden, inter, seed, str(expert), proj)
    return torch.randn(*shape, generator=g, dtype=torch.float32, device=device) * 0.02
