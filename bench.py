#!/usr/bin/env python
"""Benchmark of the routed MoE NVFP4 expert FFN (moe_forward) on GB300.

One step = one moe_forward (route, group, [quantise], gate/up + SwiGLU, down +
combine) over one batch of seeded synthetic input, inputs resident in HBM.
Default workload: decode, 4 tokens, H 4096, 128 experts, I 1536, top-8, shared
expert, W4A16, over the 10 seeded instances (seeds 0-9, each with its own
weights); step i runs instance i mod 10, so consecutive steps never share
weights and the touched weights (~0.3 GB a step, 13.6 GB in all) exceed L2.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle instead.
Multi-GPU: one process per GPU (torchrun), independent replicas, no collective
on the data path; value = tokens of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np
import torch

import synth

METRIC = "MoE NVFP4 expert-FFN tokens/s; decode HBM GB/s & prefill FP4 TFLOP/s % peak"
PROJ = ("gate", "up", "down")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"], source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, source="fallback")


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        if shutil.which("nvidia-smi") is None:
            return
        sel = str(device_index)
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            pass
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        self.f = open(self.path, "w")
        self.proc = subprocess.Popen(["nvidia-smi", "-i", sel, f"--query-gpu={self.FIELDS}",
                                      "--format=csv,noheader,nounits", "-lms", "50"],
                                     stdout=self.f, stderr=subprocess.DEVNULL)
        # let the sampler finish starting up (it opens the driver) before anything is timed
        t_end = time.time() + 10.0
        while time.time() < t_end and self.proc.poll() is None:
            self.f.flush()
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = [l.split(",") for l in open(self.path).read().strip().splitlines() if l.strip()]
        os.unlink(self.path)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- inputs

class Instance:
    """One seeded problem: device activations, router, NVFP4 weights."""

    def __init__(self, moe, w, seed, batch=0, device="cuda"):
        self.seed, self.batch = seed, batch
        self.x = synth.activations(w, seed, batch, device=device)
        self.rw = synth.router_weight(w, seed, device=device)
        self.bias = synth.router_bias(w, seed, device=device)


def build_weights(moe, w, seed):
    E, I, H = w.experts, w.inter, w.hidden
    def alloc(n, rows, cols):
        return moe.NvfpTensor(torch.empty(n, rows, cols // 2, dtype=torch.uint8, device="cuda"),
                              torch.empty(n, rows, cols // 16, dtype=torch.uint8, device="cuda"),
                              torch.empty(n, dtype=torch.float32, device="cuda"))
    shapes = {"gate": (I, H), "up": (I, H), "down": (H, I)}
    ts = {p: alloc(E, *shapes[p]) for p in PROJ}
    for e in range(E):
        for p in PROJ:
            t = ts[p]
            moe.quantize_nvfp4(synth.expert_weight(w, seed, e, p, device="cuda"),
                               out=moe.NvfpTensor(t.codes[e:e + 1], t.scales[e:e + 1], t.ts[e:e + 1]))
    routed = moe.ExpertSet(ts["gate"], ts["up"], ts["down"])
    shared = None
    if w.shared_inter:
        shared = moe.ExpertSet(*[moe.quantize_nvfp4(synth.expert_weight(w, seed, "shared", p, device="cuda"))
                                 for p in PROJ])
    return routed, shared




def ncu_traffic(key: str, workload: str):
    """DRAM bytes (read + write) of one launch of a stage's kernel, from the
    committed ncu summary table profiles/dram_traffic.txt (lines
    "stage:path workload bytes"); None when no capture covers it."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "profiles", "dram_traffic.txt")
    try:
        for line in open(path):
            f = line.split("#")[0].split()
            if len(f) >= 3 and f[0] == key and f[1] == workload:
                return int(float(f[2]))
    except OSError:
        pass
    return None


def compute_dtype(w, path):
    """The arithmetic the expert products run in: the CUDA-core engine multiplies
    dequantised weights in fp32; the tensor-core and warp-MMA engines take f16
    operands (W4A16: weights exact in f16, x scaled into range) or FP4 codes with
    E4M3 block scales (W4A4), accumulating in fp32. For AUTO this follows the
    library's rule: the tensor paths need H, I (and the shared expert's I) to be
    multiples of 256, and W4A4 takes them from 64 (token, slot) pairs on."""
    tc_ok = w.hidden % 256 == 0 and w.inter % 256 == 0 and w.shared_inter % 256 == 0
    if path == "auto":
        path = "tensor_core" if tc_ok and (w.mode == "w4a16" or w.tokens * w.top_k >= 64) else "cuda_core"
    if path == "cuda_core":
        return "fp32"
    return "f16xf16->fp32" if w.mode == "w4a16" else "fp4xfp4->fp32"


def algorithmic(w, ids_list):
    """Per-step algorithmic bytes of the gate/up and down kernels and flops,
    averaged over the instances (distinct experts touched come from routing)."""
    H, I, Is, T, k = w.hidden, w.inter, w.shared_inter, w.tokens, w.top_k
    wb = 9.0 / 16.0                                   # bytes per NVFP4 value (code nibble + 1/16 scale byte)
    act = 2.0 if w.mode == "w4a16" else wb            # activation bytes per value
    hb = 2.0 if w.mode == "w4a16" else 4.0            # SwiGLU output element as written
    gu, dn, fl = [], [], []
    for ids in ids_list:
        d = len(np.unique(ids))
        P = ids.size
        rows_s = T if Is else 0
        gu.append(d * 2 * I * H * wb + (2 * Is * H * wb if Is else 0) + T * H * act + (P * I + rows_s * Is) * hb)
        dn.append(d * H * I * wb + (H * Is * wb if Is else 0) + (P * I + rows_s * Is) * (2.0 if w.mode == "w4a16" else wb)
                  + T * H * 4)
        fl.append(2.0 * 3 * H * (P * I + rows_s * Is))
    return float(np.mean(gu)), float(np.mean(dn)), float(np.mean(fl)), float(np.mean([len(np.unique(i)) for i in ids_list]))


# ---------------------------------------------------------------- oracle (CPU)

def _draw_device():
    """Where the oracle's inputs are drawn: the GPU when there is one (the same
    bytes the GPU run uses), else the host (the reference arm needs no GPU)."""
    return "cuda" if torch.cuda.is_available() else "cpu"


class OraclePrep:
    """Host copies of one instance and the oracle's own quantisation of every
    expert it touches (untimed preparation)."""

    def __init__(self, w, inst):
        import oracle
        self.oracle, self.w = oracle, w
        self.xb = inst.x.cpu().view(torch.int16).numpy().view(np.uint16)
        self.rw = inst.rw.cpu().numpy()
        self.bias = None if inst.bias is None else inst.bias.cpu().numpy()
        self.kind = oracle.ROUTER_SIGMOID if w.router == "sigmoid" else oracle.ROUTER_SOFTMAX
        self.mode = oracle.MODE_W4A4 if w.mode == "w4a4" else oracle.MODE_W4A16
        self.route = oracle.route(self.xb, self.rw, self.bias, w.top_k, self.kind, w.renormalize)
        need = sorted(set(int(e) for e in np.unique(self.route["ids"])))
        self.packed = {e: tuple(oracle.quantize(synth.expert_weight(w, inst.seed, e, p, device=_draw_device()).cpu().numpy())
                                for p in PROJ) for e in need}
        self.shared = None
        if w.shared_inter:
            self.shared = tuple(oracle.quantize(
                synth.expert_weight(w, inst.seed, "shared", p, device=_draw_device()).cpu().numpy()) for p in PROJ)
        self.threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()

    def full(self):
        """One complete oracle moe_forward of the batch."""
        w = self.w
        self.oracle.forward(self.xb, self.rw, self.bias, lambda e: self.packed[e], k=w.top_k,
                            router_kind=self.kind, renormalize=w.renormalize, mode=self.mode, shared=self.shared)

    def pairs(self):
        """The (token, expert) pairs of the batch, then the shared expert's tokens."""
        ids = self.route["ids"]
        out = [(t, int(ids[t, j])) for t in range(ids.shape[0]) for j in range(ids.shape[1])]
        if self.shared is not None:
            out += [(t, "shared") for t in range(ids.shape[0])]
        return out

    def pair(self, t, e):
        """One complete oracle call on a one-token, one-expert problem: FFN_e(x_t)."""
        w = self.w
        packed = self.shared if e == "shared" else self.packed[e]
        self.oracle.forward(self.xb[t:t + 1], self.rw[:1], None, lambda _: packed, k=1, router_kind=self.kind,
                            renormalize=w.renormalize, mode=self.mode)


def oracle_baseline(w, inst, budget_s=15.0):
    """CPU oracle on a bounded sample: repeated full moe_forward of one batch
    (router, grouping, FP64 FFN of every touched expert), weights prepared."""
    prep = OraclePrep(w, inst)
    n, t0 = 0, time.perf_counter()
    while True:
        prep.full()
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or el * (n + 1) / n > 2 * budget_s:
            break
    desc = (f"{n} complete oracle moe_forward(s) of seed {inst.seed} ({w.tokens} tokens, "
            f"{len(prep.packed)} experts touched; FP64 numpy matmul, C router), {el:.1f} s")
    return n * w.tokens / el, desc, prep.threads


# ---------------------------------------------------------------- stage profile, roofline

def profile_stages(plan, step, n_steps):
    """Per-stage CUDA-event times (ms a launch) and kernel launches a step, from
    a separate untimed pass of n_steps steps: events recorded between two
    kernels make the second wait for the first, which would distort the timed
    region, so they are never recorded there."""
    plan.set_profiling(True)
    plan.read_profile()
    for i in range(n_steps):
        step(i)
    prof = plan.read_profile()
    plan.set_profiling(False)
    stage_ms = {k: v[0] / v[2] for k, v in prof.items() if v[2] > 0}
    launches = sum(v[1] for v in prof.values()) / n_steps
    return stage_ms, launches, n_steps


def roofline(w, stage_ms, gu_bytes, dn_bytes, flops, pk, path):
    """Roofline of the dominant stage: algorithmic bytes a launch / its mean
    event time against the measured HBM copy bandwidth; for W4A4 also its FP4
    flops against the dense NVFP4 peak (measured bf16 burst x 6, the nominal
    ratio) and the ceiling the weight bytes put on that fraction."""
    dom = max(stage_ms, key=stage_ms.get)
    alg = {"gate_up": gu_bytes, "down": dn_bytes}
    if dom not in alg:
        return None
    t = stage_ms[dom] / 1e3
    ach = alg[dom] / t / 1e9
    roof = {"kernel": dom, "bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": round(ach / pk["hbm_gbs"], 4), "traffic": ncu_traffic(f"{dom}:{path}", w.name),
            "peak_source": pk["source"], "algorithmic_bytes_per_launch": round(alg[dom]),
            "avg_launch_us": round(stage_ms[dom] * 1e3, 2)}
    if w.mode == "w4a4":
        fl = flops * (2.0 / 3.0 if dom == "gate_up" else 1.0 / 3.0)
        peak = pk["bf16_tflops"] * 6 * 1e12
        roof["fp4_tflops"] = round(fl / t / 1e12, 1)
        roof["fp4_peak_tflops"] = round(peak / 1e12, 1)
        roof["fp4_peak_source"] = "derived: measured bf16 burst x 6"
        roof["fp4_frac"] = round(fl / t / peak, 4)
        # weights alone take alg / BW: the best FP4 fraction that allows
        roof["fp4_frac_weight_bound_ceiling"] = round(min(1.0, (fl / peak) / (alg[dom] / (pk["hbm_gbs"] * 1e9))), 4)
    return roof


def run_prefill(moe, pk, args, world, local):
    """The 4096-token W4A4 prompt (H 7168, 256 experts, I 2048, top-8, sigmoid,
    Zipf bias) timed in the same run: one seeded instance, W warm-up steps,
    args.prefill_steps timed steps (each reads ~4 GB of expert weights, far more
    than L2), then an untimed per-stage pass."""
    w = synth.WORKLOADS["prompt4096_w4a4"]
    routed, shared = build_weights(moe, w, 0)
    inst = Instance(moe, w, 0)
    plan = moe.Plan(w.hidden, w.inter, w.experts, w.top_k, w.tokens, router=moe.ROUTER_SIGMOID,
                    renormalize=w.renormalize, mode=moe.W4A4, has_shared=False)
    ids = plan.route(inst.x, inst.rw, inst.bias)["topk_ids"].cpu().numpy()
    gu_bytes, dn_bytes, flops, distinct = algorithmic(w, [ids])
    out = torch.empty(w.tokens, w.hidden, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()

    def step(i):
        plan.forward(inst.x, inst.rw, inst.bias, routed, shared, out=out)

    clk = ClockSampler(local)
    for i in range(max(3, args.warmup // 2)):
        step(i)
    if plan.sync_status() != moe.OK:
        raise SystemExit("prefill moe_forward failed")
    barrier(world)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.prefill_steps):
        step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(t0.elapsed_time(t1), world) / args.prefill_steps
    clocks = clk.stop()
    if plan.sync_status() != moe.OK:
        raise SystemExit("prefill moe_forward failed")
    stage_ms, lps, n = profile_stages(plan, step, 3)
    roof = roofline(w, {k: v for k, v in stage_ms.items() if k == "gate_up"}, gu_bytes, dn_bytes, flops, pk, "auto")
    plan.close()
    return {"workload": w.name, "description": w.description, "steps": args.prefill_steps,
            "ms_per_step": round(ms, 4), "tokens_per_s": round(world * w.tokens / (ms / 1e3), 1),
            "step_fp4_tflops": round(flops / (ms / 1e3) / 1e12, 1),
            "distinct_experts": distinct, "gate_up": roof,
            "stages_us_per_step": {k: round(v * 1e3, 2) for k, v in stage_ms.items()},
            "gpu_launches_per_step": lps, "clocks": clocks,
            "l2": "inputs larger than L2: each step streams the touched experts' weights (GBs)"}


# ---------------------------------------------------------------- main arms

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    """The largest of the ranks' values (the step time every rank reports)."""
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_ours(args, w, world, rank, local):
    import moe_routed_expert_router_gb300 as moe
    moe.lib()
    pk = peaks()
    weights = {}
    insts = []
    if w.batches > 1:
        weights[w.seeds[0]] = build_weights(moe, w, w.seeds[0])
        insts = [Instance(moe, w, w.seeds[0], b) for b in range(args.instances or w.batches)]
    else:
        for s in w.seeds[:args.instances or len(w.seeds)]:
            weights[s] = build_weights(moe, w, s)
            insts.append(Instance(moe, w, s))
    plan = moe.Plan(w.hidden, w.inter, w.experts, w.top_k, w.tokens,
                    router=moe.ROUTER_SIGMOID if w.router == "sigmoid" else moe.ROUTER_SOFTMAX,
                    renormalize=w.renormalize, mode=moe.W4A4 if w.mode == "w4a4" else moe.W4A16,
                    has_shared=w.shared_inter > 0, shared_inter=w.shared_inter)
    plan.set_path({"auto": moe.PATH_AUTO, "cuda_core": moe.PATH_CUDA_CORE,
                   "tensor_core": moe.PATH_TENSOR_CORE, "warp_mma": moe.PATH_WARP_MMA}[args.path])
    ids_list = [plan.route(i.x, i.rw, i.bias)["topk_ids"].cpu().numpy() for i in insts]
    first_inst = insts[0]
    gu_bytes, dn_bytes, flops, distinct = algorithmic(w, ids_list)
    outs = [torch.empty(w.tokens, w.hidden, dtype=torch.bfloat16, device="cuda") for _ in insts]
    stream = torch.cuda.current_stream()

    def step(i):
        j = i % len(insts)
        r, s = weights[insts[j].seed]
        plan.forward(insts[j].x, insts[j].rw, insts[j].bias, r, s, out=outs[j])

    clk = ClockSampler(local)
    for i in range(args.warmup):
        step(i)
    st = plan.sync_status()
    if st != moe.OK:
        raise SystemExit(f"moe_forward failed: {moe.STATUS[st]}")
    # the timed region: K plain moe_forward calls, nothing else on the stream
    barrier(world)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = t0.elapsed_time(t1)
    st = plan.sync_status()
    if st != moe.OK:
        raise SystemExit(f"moe_forward failed: {moe.STATUS[st]}")
    ms = max_over_ranks(ms, world)
    stage_ms, launches_per_step, profiled = profile_stages(plan, step, args.profile_steps)

    # end to end through the host-buffer entry point: H2D of x + D2H of out each step
    xh = [i.x.cpu().pin_memory() for i in insts]
    oh = torch.empty(w.tokens, w.hidden, dtype=torch.bfloat16).pin_memory()

    def step_host(i):
        j = i % len(insts)
        r, s = weights[insts[j].seed]
        plan.forward_host(xh[j], insts[j].rw, insts[j].bias, r, s, oh)

    for i in range(args.warmup):
        step_host(i)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step_host(i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms_e2e = max_over_ranks(e0.elapsed_time(e1), world)
    clocks = clk.stop()

    tokens = world * args.steps * w.tokens
    value = tokens / (ms / 1e3)
    roof = roofline(w, stage_ms, gu_bytes, dn_bytes, flops, pk, args.path)
    launches = round(launches_per_step * args.steps)
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": compute_dtype(w, args.path),
        "data": "synthetic (seeded N(0,1) bf16 activations, N(0,0.02) weights quantised to NVFP4 on device)",
        "config": {"workload": w.name, "description": w.description, "tokens": w.tokens, "hidden": w.hidden,
                   "experts": w.experts, "inter": w.inter, "top_k": w.top_k, "shared_inter": w.shared_inter,
                   "mode": w.mode, "router": w.router, "instances": len(insts),
                   "l2": "inputs larger than L2: step i runs instance i mod %d with its own weights" % len(insts),
                   "parallelism": f"replicas x{world}", "distinct_experts_per_step": distinct,
                   "path": args.path},
        "e2e": {"value": round(tokens / (ms_e2e / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": w.tokens * w.hidden * 2, "d2h_bytes_per_step": w.tokens * w.hidden * 2},
        "gpu_launches": launches,
        "roofline": roof,
        "stages_us_per_step": {k: round(v * 1e3, 2) for k, v in stage_ms.items()},
        "stages_profiled_steps": profiled,
        "stages_note": "per-stage CUDA events from a separate untimed pass after the timed region",
        "hbm_gbs_whole_step": round((gu_bytes + dn_bytes) / (ms / args.steps / 1e3) / 1e9, 1),
        "clocks": clocks,
    }
    plan.close()
    del weights, insts, outs
    if args.prefill and w.name != "prompt4096_w4a4":
        res["prefill"] = run_prefill(moe, pk, args, world, local)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, desc, thr = oracle_baseline(w, first_inst, args.cpu_budget)
        res["cpu_baseline"] = {"value": round(v, 3), "unit": "tokens/s", "cores": thr, "kind": "oracle",
                               "sample": desc}
    return res


def run_reference(args, w, world, rank):
    """The oracle as it stands, on the host cores.  One step = one complete
    oracle call on one (token, expert) pair of the workload's first batch
    (cycling through the batch's routed pairs and shared-expert rows);
    tokens/s = steps / pairs-per-token / time."""
    if rank != 0:
        return None
    inst = Instance(None, w, w.seeds[0], device=_draw_device())
    prep = OraclePrep(w, inst)
    pairs = prep.pairs()
    for i in range(args.warmup):
        prep.pair(*pairs[i % len(pairs)])
    t0 = time.perf_counter()
    for i in range(args.steps):
        prep.pair(*pairs[i % len(pairs)])
    el = time.perf_counter() - t0
    per_token = w.top_k + (1 if w.shared_inter else 0)
    v = args.steps / per_token / el
    desc = (f"each step one oracle FFN call on one (token, expert) pair of seed {w.seeds[0]} "
            f"({per_token} pairs a token); {args.steps} steps in {el:.1f} s")
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "tokens": w.tokens},
            "cpu_baseline": {"value": round(v, 4), "unit": "tokens/s", "cores": prep.threads, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(v, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def relaunch(n):
    """--gpus N outside a launcher: run this same command as N replica
    processes, one a GPU, under torch.distributed.run on 127.0.0.1."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
    raise SystemExit(subprocess.call(cmd))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 2000; 200 for --impl reference, whose steps are oracle calls)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode4_w4a16", choices=list(synth.WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", default="auto", choices=["auto", "cuda_core", "tensor_core", "warp_mma"],
                    help="expert-FFN implementation (moe_plan_set_path)")
    ap.add_argument("--override", default="",
                    help="comma-separated workload fields for a scaled-down profiling run, e.g. tokens=1024,experts=64")
    ap.add_argument("--instances", type=int, default=0,
                    help="use only the first N seeded instances / batches (0 = all; for small profiling runs)")
    ap.add_argument("--profile-steps", type=int, default=32,
                    help="steps of the untimed per-stage pass after the timed region")
    ap.add_argument("--prefill-steps", type=int, default=10,
                    help="timed steps of the 4096-token W4A4 prompt sub-record")
    ap.add_argument("--no-prefill", dest="prefill", action="store_false",
                    help="skip the 4096-token W4A4 prompt sub-record")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    w = synth.WORKLOADS[args.workload]
    if args.override:
        kv = dict(item.split("=") for item in args.override.split(","))
        w = synth.scaled(w, **{k: int(v) for k, v in kv.items()})
    if args.steps is None:
        args.steps = 200 if args.impl == "reference" else 2000
    if args.impl == "reference":
        world, rank = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0"))
        if rank == 0:
            torch.cuda.set_device(0) if torch.cuda.is_available() else None
            res = run_reference(args, w, world, rank)
            print(json.dumps(res), flush=True)
        return
    if args.gpus > 1 and int(os.environ.get("WORLD_SIZE", "1")) == 1:
        relaunch(args.gpus)
    if args.gpus != int(os.environ.get("WORLD_SIZE", "1")):
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={os.environ.get('WORLD_SIZE')}")
    world, rank, local = dist_init()
    res = run_ours(args, w, world, rank, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
