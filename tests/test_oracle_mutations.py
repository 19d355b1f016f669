"""Mutation checks of the oracle's pins (no GPU).

Each test plants one plausible mistake in the oracle, on the CPU, and requires
that the pins which guard that part of it fail:
  * codes unpacked with the nibbles swapped (element 2i read from bits 4..7);
  * an expert offset off by one;
  * the last pairs of the last expert's segment dropped (a lost last tile);
  * the per-expert tensor scale left out of the dequantisation;
  * MXFP4 block scales applied to 16-value blocks.
The mistakes are planted by replacing a function of the oracle module for the
duration of one test (monkeypatch); nothing here touches the CUDA path."""
import numpy as np
import pytest

import oracle
import test_oracle_ffn as ffn
import test_oracle_quant as quant
import test_oracle_router as router

_unpack, _group, _dequantize = oracle.unpack_codes, oracle.group, oracle.dequantize


def _swapped_unpack(codes):
    q = _unpack(codes)
    q[..., 0::2], q[..., 1::2] = q[..., 1::2].copy(), q[..., 0::2].copy()
    return q


def _offset_off_by_one(ids, E):
    offsets, rows = _group(ids, E)
    offsets = offsets.copy()
    if E > 1:
        offsets[1] = min(offsets[1] + 1, offsets[-1])
    return offsets, rows


def _last_pairs_dropped(ids, E):
    offsets, rows = _group(ids, E)
    offsets = offsets.copy()
    last = int(np.nonzero(np.diff(offsets))[0][-1])      # last expert with pairs
    offsets[last + 1:] -= 1                              # its final pair is never computed
    return offsets, rows


def _no_tensor_scale(codes, scales, ts):
    return _dequantize(codes, scales, 1.0)


def _fails(fn, *a):
    """The pin turns red: an assertion fails, or an expert it checks is missing."""
    with pytest.raises((AssertionError, KeyError)):
        fn(*a)


def test_the_pins_pass_unmutated():
    ffn.test_hand_worked_one_token_two_experts()
    ffn.test_w4a4_hand_worked_swiglu_tensor_scales()
    ffn.test_single_expert_is_a_dense_swiglu_mlp()
    quant.test_hand_worked_blocks()
    router.test_group_is_a_stable_sort()
    router.test_route_permutation_covers_every_pair_once()


def test_swapped_nibbles_are_caught(monkeypatch):
    monkeypatch.setattr(oracle, "unpack_codes", _swapped_unpack)
    _fails(quant.test_hand_worked_blocks)
    _fails(ffn.test_hand_worked_one_token_two_experts)
    _fails(ffn.test_w4a4_hand_worked_swiglu_tensor_scales)


def test_off_by_one_expert_offset_is_caught(monkeypatch):
    monkeypatch.setattr(oracle, "group", _offset_off_by_one)
    _fails(router.test_group_is_a_stable_sort)
    _fails(ffn.test_hand_worked_one_token_two_experts)
    _fails(router.test_route_permutation_covers_every_pair_once)


def test_dropped_last_tile_is_caught(monkeypatch):
    monkeypatch.setattr(oracle, "group", _last_pairs_dropped)
    _fails(router.test_group_is_a_stable_sort)
    _fails(ffn.test_single_expert_is_a_dense_swiglu_mlp)
    _fails(ffn.test_w4a4_hand_worked_swiglu_tensor_scales)


def test_missing_tensor_scale_is_caught(monkeypatch):
    monkeypatch.setattr(oracle, "dequantize", _no_tensor_scale)
    _fails(ffn.test_hand_worked_one_token_two_experts)
    _fails(ffn.test_w4a4_hand_worked_swiglu_tensor_scales)


def test_mx_scale_block_of_the_wrong_size_is_caught(monkeypatch):
    import test_oracle_mx as mx
    def bad(codes, scales):   # each scale applied to 16 values, the row's scales then reused
        s16 = np.repeat(oracle.e8m0_table()[np.asarray(scales, np.uint8)], 16, axis=-1)
        return oracle.e2m1_table()[oracle.unpack_codes(codes)] * np.concatenate([s16, s16], axis=-1)
    monkeypatch.setattr(oracle, "dequantize_mx", bad)
    _fails(mx.test_error_bound_and_clipping)
    _fails(mx.test_quantiser_is_idempotent_on_its_grid)
