"""Planted mistakes in the oracle (CPU only): each plausible error must make at
least one pin in test_oracle_pins.py fail.  The mutation is applied with
monkeypatch for the duration of one check and undone afterwards."""

import numpy as np

import oracle
import oracle.moe_oracle as M
from tests import test_oracle_pins as P


def patch(monkeypatch, name, fn):
    """Replace an oracle function everywhere it is reachable: the module the
    oracle's own functions call into, and the package namespace the pins use."""
    monkeypatch.setattr(M, name, fn)
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, fn)


def fails(check):
    try:
        check()
    except AssertionError:
        return True
    return False


def test_silu_without_sigmoid_is_caught(monkeypatch):
    patch(monkeypatch, "silu", lambda z: np.asarray(z, np.float64))
    assert fails(P.test_silu_closed_form) or fails(P.test_grouped_gemm_matches_per_token_loops)
    assert fails(P.test_grouped_gemm_matches_per_token_loops)


def test_swapped_w1_w3_roles_are_caught(monkeypatch):
    orig = M.expert_swiglu

    def swapped(a, w1, w3, w2):
        return orig(a, w3, w1, w2)
    patch(monkeypatch, "expert_swiglu", swapped)
    assert fails(P.test_grouped_gemm_matches_per_token_loops)
    assert fails(P.test_grouped_gemm_single_expert_is_dense_swiglu)


def test_transposed_router_is_caught(monkeypatch):
    def wrong(x, wg, gate_bias=None):
        out = np.asarray(x, np.float64) @ np.asarray(wg, np.float64)[:, :np.asarray(x).shape[1]].T
        return out
    patch(monkeypatch, "router_logits", wrong)
    assert fails(P.test_router_matches_brute_force)


def test_dropped_gate_bias_is_caught(monkeypatch):
    orig = M.router_logits
    patch(monkeypatch, "router_logits", lambda x, wg, gate_bias=None: orig(x, wg))
    assert fails(P.test_router_matches_brute_force)
    assert fails(P.test_router_integer_inputs_exact)


def test_highest_index_tie_break_is_caught(monkeypatch):
    def wrong_order(keys_row):
        k = -np.asarray(keys_row)
        idx = np.arange(len(k))
        return np.lexsort((-idx, k))          # equal keys: higher index first
    patch(monkeypatch, "_order_desc_low_index", wrong_order)
    assert fails(P.test_softmax_topk_golden_ties)


def test_missing_renormalisation_is_caught(monkeypatch):
    def no_renorm(logits, E, K):
        lg = np.asarray(logits)[:, :E]
        ids = np.argsort(-lg, axis=1, kind="stable")[:, :K].astype(np.int32)
        p = np.exp(lg - lg.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        return ids, np.take_along_axis(p, ids, 1)
    patch(monkeypatch, "topk_softmax_renorm", no_renorm)
    assert fails(P.test_softmax_topk_golden_closed_form)


def test_biased_sigmoid_weights_are_caught(monkeypatch):
    def biased(logits_f32, sel_bias, E, K, scale):
        lg = np.asarray(logits_f32, np.float32)[:, :E]
        s = M.sigmoid_f32(lg)
        key = (s + np.asarray(sel_bias, np.float32)[None, :]).astype(np.float32)
        ids = np.argsort(-key, axis=1, kind="stable")[:, :K].astype(np.int32)
        ks = np.take_along_axis(key, ids, 1).astype(np.float64)   # mistake: biased keys as weights
        return ids, scale * ks / ks.sum(1, keepdims=True)
    patch(monkeypatch, "topk_sigmoid_bias", biased)
    assert fails(P.test_sigmoid_bias_golden_closed_form)


def test_wrong_exp_constant_is_caught(monkeypatch):
    patch(monkeypatch, "_LN2_LO", np.float32(0.0))      # Cody-Waite tail dropped
    assert fails(P.test_exp_f32_accuracy_and_special_values)


def test_unstable_permute_is_caught(monkeypatch):
    def unstable(ids, E):
        flat = np.asarray(ids, dtype=np.int64).ravel()
        counts = np.bincount(flat, minlength=E)[:E]
        offsets = np.zeros(E + 1, dtype=np.int64)
        offsets[1:] = np.cumsum(counts)
        r2f = np.argsort(flat * (flat.size + 1) - np.arange(flat.size), kind="stable")  # reversed ties
        f2r = np.empty_like(r2f)
        f2r[r2f] = np.arange(flat.size)
        return offsets.astype(np.int32), r2f.astype(np.int32), f2r.astype(np.int32)
    patch(monkeypatch, "permute", unstable)
    assert fails(P.test_permute_golden_worked_example)


def test_off_by_one_offsets_are_caught(monkeypatch):
    orig = M.permute

    def shifted(ids, E):
        off, r2f, f2r = orig(ids, E)
        off = off.copy()
        off[1:-1] += 1
        return off, r2f, f2r
    patch(monkeypatch, "permute", shifted)
    assert fails(P.test_permute_golden_worked_example)


def test_missing_shared_expert_gate_is_caught(monkeypatch):
    orig = M.unpermute

    def ungated(y, f2r, w, T, K, shared_y=None, g_sh=None):
        return orig(y, f2r, w, T, K, shared_y, None if g_sh is None else np.ones_like(g_sh))
    patch(monkeypatch, "unpermute", ungated)
    assert fails(P.test_unpermute_adds_gated_shared_expert)


def test_wrong_fp8_block_index_is_caught(monkeypatch):
    orig = M.dequant_fp8_block

    def transposed_scales(codes, scales, block=128):
        s = np.asarray(scales)
        return orig(codes, np.swapaxes(s, -1, -2) if s.shape[-1] == s.shape[-2] else s, block)
    patch(monkeypatch, "dequant_fp8_block", transposed_scales)
    assert fails(P.test_dequant_block_layout_with_ragged_tail)


def test_wrong_e4m3_bias_is_caught(monkeypatch):
    table = np.array([M._e4m3_value(c) * (2.0 if (c & 0x78) else 1.0) for c in range(256)])
    patch(monkeypatch, "_E4M3_TABLE", table)
    assert fails(P.test_e4m3_known_codes)
    assert fails(P.test_e4m3_all_codes_match_torch)


def test_swapped_mxfp4_nibbles_are_caught(monkeypatch):
    real = M.dequant_mxfp4

    def swapped(packed, scales, block=32):
        b = np.asarray(packed, np.uint8)
        return real(((b & 0xF) << 4) | (b >> 4), scales, block)
    patch(monkeypatch, "dequant_mxfp4", swapped)
    assert fails(P.test_mxfp4_golden_worked_example)


def test_mxfp4_scale_off_by_one_is_caught(monkeypatch):
    real = M.dequant_mxfp4
    patch(monkeypatch, "dequant_mxfp4",
          lambda packed, scales, block=32: real(packed, np.asarray(scales, np.uint8) + 1, block))
    assert fails(P.test_mxfp4_golden_worked_example)
    assert fails(P.test_mxfp4_scale_is_a_power_of_two_per_32_elements)


def test_w8a8_ties_away_from_zero_are_caught(monkeypatch):
    orig = M.e4m3_round

    def away(v):
        v = np.asarray(v, np.float64)
        c = orig(v)
        # at an exact midpoint take the larger magnitude instead of the even code
        up = orig(np.nextafter(np.abs(v), np.inf) * np.sign(v))
        mid = (orig(np.nextafter(np.abs(v), 0) * np.sign(v)) != up) & (c != up)
        return np.where(mid, up, c).astype(np.uint8)
    patch(monkeypatch, "e4m3_round", away)
    assert fails(P.test_e4m3_round_matches_torch_cast)


def test_w8a8_scale_block_of_64_is_caught(monkeypatch):
    orig = M.quantize_act_fp8
    patch(monkeypatch, "quantize_act_fp8", lambda a, block=128: orig(a, 64))
    assert fails(P.test_quantize_act_fp8_closed_forms)
    assert fails(P.test_quantize_act_fp8_matches_brute_force)


def test_w8a8_scale_over_240_is_caught(monkeypatch):
    # a wrong largest code (240, the e4m3 maximum of another convention)
    def q240(a, block=128):
        a32 = np.asarray(a, np.float32)
        nb = -(-a32.shape[1] // block)
        codes = np.zeros(a32.shape, np.uint8)
        sc = np.zeros((a32.shape[0], nb), np.float32)
        for j in range(nb):
            blk = a32[:, j * block:(j + 1) * block]
            sb = (np.abs(blk).max(axis=1) / np.float32(240.0)).astype(np.float32)
            safe = np.where(sb > 0, sb, np.float32(1.0)).astype(np.float32)
            c = M.e4m3_round((blk / safe[:, None]).astype(np.float32))
            c[sb == 0] = 0
            codes[:, j * block:(j + 1) * block] = c
            sc[:, j] = sb
        return codes, sc
    patch(monkeypatch, "quantize_act_fp8", q240)
    assert fails(P.test_quantize_act_fp8_closed_forms)
    assert fails(P.test_quantize_act_fp8_matches_brute_force)


def test_w8a8_unrounded_hact_is_caught(monkeypatch):
    patch(monkeypatch, "round_bf16", lambda v: np.asarray(v, np.float64))
    assert fails(P.test_round_bf16_matches_torch)
    assert fails(P.test_grouped_gemm_w8a8_matches_brute_force)


def test_w8a8_unquantised_second_gemm_is_caught(monkeypatch):
    orig_gg = M.grouped_gemm_w8a8

    def no_second(xp, offsets, w1, w3, w2):
        hact, _ = orig_gg(xp, offsets, w1, w3, w2)
        y = np.zeros((hact.shape[0], w2.shape[1]))
        for e in range(len(offsets) - 1):
            lo, hi = int(offsets[e]), int(offsets[e + 1])
            y[lo:hi] = hact[lo:hi] @ np.asarray(w2[e], np.float64).T
        return hact, y
    patch(monkeypatch, "grouped_gemm_w8a8", no_second)
    assert fails(P.test_grouped_gemm_w8a8_matches_brute_force)
