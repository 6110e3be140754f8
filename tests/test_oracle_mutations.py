"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in the oracle (on the CPU, by replacing one
oracle function for the duration of the test) and checks that a pin of
tests/test_oracle_pins.py then fails: a wrong nibble order, a dropped zero
point, the wrong rounding mode or scale in the quantiser, a wrong group
index, a swapped gate/up or a wrong activation in SwiGLU (in the layer and in
its SwiGLU stage), a transposed down-stage weight, ties broken the other way or unnormalised weights in the router, a mis-weighted shared
expert.
"""

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins


def fails(fn, *args):
    with pytest.raises(AssertionError):
        fn(*args)


def test_pack_high_nibble_first_is_caught(monkeypatch, golden_dir):
    def pack_reversed(nib):
        nib = np.asarray(nib, dtype=np.uint32)
        N, K = nib.shape
        n = nib.reshape(N, K // 8, 8)
        word = np.zeros((N, K // 8), dtype=np.uint32)
        for j in range(8):
            word |= n[:, :, j] << np.uint32(4 * (7 - j))
        return word.view(np.int32)
    monkeypatch.setattr(oracle, "pack_nibbles", pack_reversed)
    fails(pins.test_pack_matches_hand_derived_words, golden_dir)
    fails(pins.test_pack_random_against_python_ints)


def test_dropped_zero_point_is_caught(monkeypatch):
    def dequant_no_zero_point(qw, sc, group=32):
        q = oracle.unpack_nibbles(qw).astype(np.float32)
        return (q * np.repeat(sc, group, axis=1)).astype(np.float32)
    monkeypatch.setattr(oracle, "dequantize", dequant_no_zero_point)
    fails(pins.test_dequant_closed_form_all_nibbles)


def test_round_half_away_from_zero_is_caught(monkeypatch, golden_dir):
    real_rint = np.rint

    class NpWithAwayRounding:
        def __getattr__(self, name):
            return getattr(np, name)

        @staticmethod
        def rint(v):
            return np.sign(v) * np.floor(np.abs(v) + 0.5)

    monkeypatch.setattr(oracle, "np", NpWithAwayRounding())
    try:
        fails(pins.test_quantizer_hand_cases, golden_dir)
    finally:
        assert np.rint is real_rint


def test_wrong_scale_divisor_is_caught(monkeypatch):
    def quantize_over_8(w, group=32):  # s = max|w| / 8, codes clamped as usual
        w = np.ascontiguousarray(w, dtype=np.float32)
        N, K = w.shape
        wg = w.reshape(N, K // group, group)
        s = (np.abs(wg).max(axis=2) / np.float32(8)).astype(np.float32)
        safe = np.where(s > 0, s, np.float32(1.0)).astype(np.float32)
        q = np.rint((wg / safe[:, :, None]).astype(np.float32))
        q = np.clip(np.where(s[:, :, None] > 0, q, 0.0), -8, 7).astype(np.int64)
        return oracle.pack_nibbles((q + 8).reshape(N, K)), s
    monkeypatch.setattr(oracle, "quantize_w4a16", quantize_over_8)
    fails(pins.test_quantizer_roundtrip_bound_and_extremes)


def test_wrong_group_index_is_caught(monkeypatch):
    real = oracle.dequantize

    def dequant_first_group_only(qw, sc, group=32):
        return real(qw, np.repeat(sc[:, :1], sc.shape[1], axis=1), group)
    monkeypatch.setattr(oracle, "dequantize", dequant_first_group_only)
    fails(pins.test_gemm_matches_exact_triple_loop, 2, 5, 64)


def test_wrong_swiglu_is_caught(monkeypatch):
    monkeypatch.setattr(oracle, "silu", lambda g: np.asarray(g, dtype=np.float64))
    fails(pins.test_moe_ref_top1_unit_weight_is_two_gemms_and_swiglu)
    fails(pins.test_silu_closed_forms)


def test_router_ties_to_higher_id_are_caught(monkeypatch):
    real = oracle.moe_route_ref

    def route_ties_high(x, router_w, bias, topk, route_scale):
        logits, bound, _, _ = real(x, router_w, bias, topk, route_scale)
        s = oracle.sigmoid(logits)
        b = np.zeros(s.shape[1]) if bias is None else np.asarray(bias, np.float64)
        sel = s + b
        ids = np.zeros((s.shape[0], topk), np.int32)
        w = np.zeros((s.shape[0], topk))
        for t in range(s.shape[0]):
            order = sorted(range(s.shape[1]), key=lambda e: (-sel[t, e], -e))[:topk]
            ids[t] = order
            w[t] = route_scale * s[t, order] / s[t, order].sum()
        return logits, bound, ids, w
    monkeypatch.setattr(oracle, "moe_route_ref", route_ties_high)
    fails(pins.test_route_ties_bias_and_full_selection)


def test_unnormalised_router_weights_are_caught(monkeypatch):
    real = oracle.moe_route_ref

    def route_unnormalised(x, router_w, bias, topk, route_scale):
        logits, bound, ids, w = real(x, router_w, bias, topk, route_scale)
        s = oracle.sigmoid(logits)
        return logits, bound, ids, route_scale * np.take_along_axis(s, ids.astype(np.int64), 1)
    monkeypatch.setattr(oracle, "moe_route_ref", route_unnormalised)
    fails(pins.test_route_against_brute_force, 4, 7, 16, 3, False)


def test_misweighted_shared_expert_is_caught(monkeypatch):
    real = oracle.moe_ref

    def moe_ref_half_last_slot(x, ids, rw, *a, **k):
        rw = np.array(rw, dtype=np.float64)
        if rw.shape[1] > 1:
            rw[:, -1] *= 0.5
        return real(x, ids, rw, *a, **k)
    monkeypatch.setattr(oracle, "moe_ref", moe_ref_half_last_slot)
    fails(pins.test_moe_block_shared_expert_closed_forms)


def test_down_stage_transposed_weight_is_caught(monkeypatch):
    real_deq = oracle.dequantize

    def down_transposed(h_in, route_w, qw_dn, sc_dn, eps, group=32):
        h_in = np.asarray(h_in, dtype=np.float64)
        r = np.asarray(route_w, dtype=np.float32).astype(np.float64)
        w = real_deq(qw_dn, sc_dn, group).astype(np.float64)
        o = r[:, None] * (h_in @ w)          # W instead of W^T
        return o, np.abs(o)
    monkeypatch.setattr(oracle, "moe_down_ref", down_transposed)
    fails(pins.test_moe_down_stage_matches_brute_force_and_scales)


def test_swiglu_stage_gate_up_swapped_is_caught(monkeypatch):
    real_deq = oracle.dequantize

    def swiglu_swapped(x, qw_gu, sc_gu, bf16_mode, eps, group=32):
        w = real_deq(qw_gu, sc_gu, group).astype(np.float64)
        I = w.shape[0] // 2
        gu = np.asarray(x, dtype=np.float64) @ w.T
        h = oracle.silu(gu[:, I:]) * gu[:, :I]   # silu(up) * gate
        return h, np.abs(h) + 1.0
    monkeypatch.setattr(oracle, "moe_swiglu_ref", swiglu_swapped)
    fails(pins.test_moe_swiglu_stage_matches_brute_force)
