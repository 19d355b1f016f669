"""Host logic of bench.py, no GPU: the timing reduction over ranks (two gloo
ranks), the DRAM-traffic table lookup, the compute-type label and the
algorithmic byte count."""
import importlib.util
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    b = _bench()
    b.barrier(world)
    out[rank] = b.max_over_ranks(1.5 + 2.0 * rank, world)   # rank 1 is the slower one
    b.barrier(world)
    dist.destroy_process_group()


def test_step_time_is_the_max_over_two_gloo_ranks():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    assert dict(out) == {0: 3.5, 1: 3.5}


def test_single_rank_needs_no_process_group():
    assert _bench().max_over_ranks(2.25, 1) == 2.25


@pytest.mark.parametrize("name", ["decode4_w4a16", "verify16_w4a4", "prompt512_w4a16", "prompt4096_w4a4"])
def test_traffic_table_covers_each_bench_workload(name):
    b = _bench()
    for stage in ("gate_up", "down"):
        v = b.ncu_traffic(f"{stage}:auto", name)
        assert v is not None and v > 10 * 2**20, (stage, name, v)
    assert b.ncu_traffic("gate_up:auto", "no_such_workload") is None


def test_compute_type_label_follows_the_engine_choice():
    b = _bench()
    W = synth.WORKLOADS
    assert b.compute_dtype(W["decode4_w4a16"], "auto") == "f16xf16->fp32"
    assert b.compute_dtype(W["prompt4096_w4a4"], "auto") == "fp4xfp4->fp32"
    assert b.compute_dtype(W["tiny_w4a16"], "auto") == "fp32"          # I = 128: no tensor path
    assert b.compute_dtype(W["decode4_w4a16"], "cuda_core") == "fp32"
    small = synth.scaled(W["verify16_w4a4"], tokens=4)                  # 32 pairs: below the W4A4 tensor path
    assert b.compute_dtype(small, "auto") == "fp32"


def test_algorithmic_bytes_count_each_touched_expert_once():
    b = _bench()
    w = synth.scaled(synth.WORKLOADS["decode4_w4a16"], tokens=2, top_k=2, shared_inter=0)
    H, I = w.hidden, w.inter
    two = np.array([[3, 5], [5, 3]])            # both tokens on experts 3 and 5
    three = np.array([[3, 5], [7, 3]])          # three experts touched
    g1, d1, f1, n1 = b.algorithmic(w, [two])
    g2, d2, f2, n2 = b.algorithmic(w, [three])
    assert (n1, n2) == (2, 3)
    assert g2 - g1 == pytest.approx(2 * I * H * 9 / 16)   # one more expert's gate and up weights
    assert d2 - d1 == pytest.approx(H * I * 9 / 16)       # and its down weights
    assert f1 == f2                                        # flops follow the pairs, not the experts
