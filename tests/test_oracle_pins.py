"""Pins for the CPU oracle: brute force, closed forms, library routines and
invariants -- none of them re-types the oracle's own formulas."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_07_gb300 import synth
from tests import brute

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- formats

def test_bf16_known_codes():
    codes = np.array([0x3F80, 0xC000, 0x4049, 0x0000, 0x8000, 0x7F7F, 0x0001], np.uint16)
    want = [1.0, -2.0, 3.140625, 0.0, -0.0, 3.3895313892515355e38, 2.0 ** -133]
    got = oracle.bf16_to_f64(codes)
    assert list(got) == want
    assert math.copysign(1.0, got[4]) == -1.0


def test_bf16_all_codes_match_torch():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = oracle.bf16_to_f64(codes)
    ok = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[ok], ref[ok])


def test_e4m3_known_codes():
    got = oracle.e4m3_to_f64(np.array([0x38, 0x7E, 0x08, 0x01, 0xB8, 0x00, 0x07, 0x40], np.uint8))
    assert list(got) == [1.0, 448.0, 2.0 ** -6, 2.0 ** -9, -1.0, 0.0, 7 * 2.0 ** -9, 2.0]
    assert np.isnan(oracle.e4m3_to_f64(np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    got = oracle.e4m3_to_f64(codes)
    ok = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[ok], ref[ok])


def test_dequant_block_layout_with_ragged_tail():
    # codes all 1.0; each 128x128 block gets its own scale, last blocks 64/72 wide
    rows, cols = 192, 200
    codes = np.full((rows, cols), 0x38, np.uint8)
    scales = np.array([[2.0, 3.0], [5.0, 7.0]], np.float32)
    w = oracle.dequant_fp8_block(codes, scales)
    assert w[0, 0] == 2.0 and w[127, 127] == 2.0
    assert w[0, 128] == 3.0 and w[127, 199] == 3.0
    assert w[128, 0] == 5.0 and w[191, 127] == 5.0
    assert w[128, 128] == 7.0 and w[191, 199] == 7.0
    # a batch of experts keeps its own scale grid
    w3 = oracle.dequant_fp8_block(np.stack([codes, codes]), np.stack([scales, 2 * scales]))
    assert w3[1, 191, 199] == 14.0


def test_dequant_matches_synth_quantisation_error_bound():
    w = rng(0).standard_normal((130, 260)).astype(np.float32)
    q, s = synth.quantize_fp8_block(w)
    d = oracle.dequant_fp8_block(q, s)
    # e4m3 has 3 mantissa bits: |w - d| <= 2^-4 |w| for normals, plus the
    # subnormal spacing 2^-9 * scale near zero
    bound = 2.0 ** -4 * np.abs(w) + 2.0 ** -10 * np.repeat(np.repeat(s, 128, 0), 128, 1)[:130, :260]
    assert np.all(np.abs(d - w) <= bound + 1e-12)


# ---------------------------------------------------------------- router

def test_router_matches_brute_force():
    r = rng(1)
    x = r.standard_normal((3, 7))
    wg = r.standard_normal((5, 7))
    b = r.standard_normal(5)
    want = np.array(brute.router(x.tolist(), wg.tolist(), b.tolist()))
    assert np.allclose(oracle.router_logits(x, wg, b), want, rtol=0, atol=1e-12)
    want0 = np.array(brute.router(x.tolist(), wg.tolist()))
    assert np.allclose(oracle.router_logits(x, wg), want0, rtol=0, atol=1e-12)


def test_router_one_hot_rows_pick_weight_columns():
    H, G = 6, 4
    wg = rng(2).standard_normal((G, H))
    x = np.eye(H)[[3, 0, 5]]
    out = oracle.router_logits(x, wg)
    assert np.array_equal(out, wg[:, [3, 0, 5]].T)


def test_router_integer_inputs_exact():
    x = np.array([[1, 2, 3, 4], [0, -1, 0, 2]], np.float64)
    wg = np.array([[1, 0, 0, 1], [2, 2, 2, 2], [-1, 1, -1, 1]], np.float64)
    assert np.array_equal(oracle.router_logits(x, wg, [0.5, 0, 0]),
                          [[5.5, 20, 2], [2.5, 2, 1]])


# ---------------------------------------------------------------- routing

def test_softmax_topk_golden_closed_form():
    g = gold("route_softmax_ln.json")
    lg = np.log(np.array([g["logits_ln_of"]], np.float64))
    ids, w = oracle.topk_softmax_renorm(lg, g["E"], g["K"])
    assert ids[0].tolist() == g["ids"]
    assert np.allclose(w[0], np.array(g["weights_num"]) / g["weights_den"], rtol=1e-14)


def test_softmax_topk_golden_ties():
    for case in gold("route_ties.json")["cases"]:
        lg = np.array([case["logits"]], np.float64)
        ids, w = oracle.topk_softmax_renorm(lg, lg.shape[1], case["K"])
        assert ids[0].tolist() == case["ids"]
        assert np.allclose(w[0], case["weights"], rtol=1e-14)


def test_softmax_topk_matches_brute_force():
    r = rng(3)
    T, E, K = 25, 9, 3
    lg = r.standard_normal((T, E + 1))
    ids, w = oracle.topk_softmax_renorm(lg, E, K)
    for t in range(T):
        sel, ww = brute.softmax_renorm_row(lg[t].tolist(), E, K)
        assert ids[t].tolist() == sel
        assert np.allclose(w[t], ww, rtol=1e-13)


def test_softmax_topk_k_equals_e_is_full_softmax():
    lg = rng(4).standard_normal((4, 6))
    ids, w = oracle.topk_softmax_renorm(lg, 6, 6)
    full = torch.softmax(torch.from_numpy(lg), dim=1).numpy()
    for t in range(4):
        assert sorted(ids[t].tolist()) == list(range(6))
        assert np.allclose(w[t], full[t, ids[t]], rtol=1e-13)
        assert abs(w[t].sum() - 1.0) < 1e-14


def test_softmax_topk_ignores_shared_gate_column():
    lg = np.zeros((1, 5))
    lg[0, 4] = 100.0           # column E = 4 is the shared gate
    lg[0, 2] = 1.0
    ids, _ = oracle.topk_softmax_renorm(lg, 4, 1)
    assert ids[0, 0] == 2


def test_exp_f32_accuracy_and_special_values():
    z = np.linspace(-87.0, 88.0, 200001).astype(np.float32)
    got = oracle.moe_oracle._exp_f32_reduced(z).astype(np.float64)
    ref = np.exp(z.astype(np.float64))
    rel = np.abs(got - ref) / ref
    assert rel.max() < 2.5 * 2.0 ** -24 * 2  # within ~2 ulp of the exact value
    assert oracle.moe_oracle._exp_f32_reduced(np.float32([0.0]))[0] == np.float32(1.0)


def test_sigmoid_f32_accuracy_and_special_values():
    l = np.linspace(-30, 30, 120001).astype(np.float32)
    got = oracle.sigmoid_f32(l).astype(np.float64)
    ref = 1.0 / (1.0 + np.exp(-l.astype(np.float64)))
    assert (np.abs(got - ref) / ref).max() < 4 * 2.0 ** -24
    s = oracle.sigmoid_f32(np.float32([0.0, 100.0, -100.0, 88.5, -88.5]))
    assert s.tolist() == [0.5, 1.0, 0.0, 1.0, 0.0]
    assert s.dtype == np.float32


def test_sigmoid_bias_golden_closed_form():
    g = gold("route_sigmoid_bias.json")
    lg = (np.array([g["logits_ln3_multiple"]], np.float64) * math.log(3.0)).astype(np.float32)
    for case in g["cases"]:
        ids, w = oracle.topk_sigmoid_bias(lg, np.array(g["bias"], np.float32), 4, case["K"],
                                          g["scale"])
        assert ids[0].tolist() == case["ids"]
        want = (case["weights"] if "weights" in case
                else np.array(case["weights_num"]) / case["weights_den"])
        assert np.allclose(w[0], want, rtol=1e-6)
        assert abs(w[0].sum() - g["scale"]) < 1e-12


def test_sigmoid_bias_matches_brute_force():
    r = rng(5)
    T, E, K, scale = 40, 24, 5, 2.5
    lg = r.standard_normal((T, E)).astype(np.float32)
    b = (r.standard_normal(E) * 0.3).astype(np.float32)
    ids, w = oracle.topk_sigmoid_bias(lg, b, E, K, scale)
    checked = 0
    for t in range(T):
        keys = sorted(brute.sigmoid(float(lg[t, e])) + float(b[e]) for e in range(E))
        if keys[-K] - keys[-K - 1] < 1e-5:
            continue  # a near tie at the K-th place: float32 keys may order it otherwise
        sel, ww = brute.sigmoid_bias_row(lg[t].astype(np.float64).tolist(), b.tolist(), E, K, scale)
        assert ids[t].tolist() == sel
        assert np.allclose(w[t], ww, rtol=1e-6)
        checked += 1
    assert checked >= T - 3


def test_shared_gate_closed_form():
    lg = np.array([[9.0, 0.0], [9.0, math.log(3.0)], [9.0, -math.log(3.0)]])
    assert np.allclose(oracle.shared_gate(lg, 1), [0.5, 0.75, 0.25], rtol=1e-15)


# ---------------------------------------------------------------- permute

def test_permute_golden_worked_example():
    g = gold("permute_worked.json")
    off, r2f, f2r = oracle.permute(np.array(g["ids"]), g["E"])
    assert off.tolist() == g["offsets"]
    assert r2f.tolist() == g["row_to_flat"]
    assert f2r.tolist() == g["flat_to_row"]


@pytest.mark.parametrize("T,K,E", [(37, 3, 11), (1, 1, 1), (5, 4, 4), (64, 8, 128)])
def test_permute_matches_brute_force_and_is_a_bijection(T, K, E):
    ids = synth.random_ids(T, K, E, seed=T)
    off, r2f, f2r = oracle.permute(ids, E)
    b_off, b_r2f, b_f2r = brute.permute(ids.ravel().tolist(), E)
    assert off.tolist() == b_off and r2f.tolist() == b_r2f and f2r.tolist() == b_f2r
    R = T * K
    assert sorted(r2f.tolist()) == list(range(R))
    assert np.array_equal(f2r[r2f], np.arange(R))
    assert off[0] == 0 and off[-1] == R and np.all(np.diff(off) >= 0)


def test_permute_empty_experts_repeat_offsets():
    ids = np.array([[0, 3], [3, 0]])
    off, _, _ = oracle.permute(ids, 5)
    assert off.tolist() == [0, 2, 2, 2, 4, 4]


def test_gather_rows():
    x = np.arange(12.0).reshape(3, 4)
    ids = np.array([[1, 0], [0, 1], [1, 1]])
    _, r2f, _ = oracle.permute(ids, 2)
    xp = oracle.gather_rows(x, r2f, 2)
    # expert 0 gets replicas f=1 (t0), f=2 (t1); expert 1 gets f=0,3,4,5
    assert np.array_equal(xp, x[[0, 1, 0, 1, 2, 2]])


# ---------------------------------------------------------------- experts

def test_silu_closed_form():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-15
    assert abs(oracle.silu(-math.log(3.0)) + 0.25 * math.log(3.0)) < 1e-15


def test_grouped_gemm_matches_per_token_loops():
    r = rng(6)
    E, H, I, T, K = 3, 6, 4, 5, 2
    x = r.standard_normal((T, H))
    w1, w3 = r.standard_normal((E, I, H)), r.standard_normal((E, I, H))
    w2 = r.standard_normal((E, H, I))
    ids = synth.random_ids(T, K, E, seed=7)
    off, r2f, _ = oracle.permute(ids, E)
    xp = oracle.gather_rows(x, r2f, K)
    hact, y = oracle.grouped_gemm(xp, off, w1, w3, w2)
    for row, f in enumerate(r2f):
        e = ids.ravel()[f]
        hb, yb = brute.swiglu_token(x[f // K].tolist(), w1[e].tolist(), w3[e].tolist(),
                                    w2[e].tolist())
        assert np.allclose(hact[row], hb, rtol=1e-12, atol=1e-12)
        assert np.allclose(y[row], yb, rtol=1e-12, atol=1e-12)


def test_grouped_gemm_single_expert_is_dense_swiglu():
    r = rng(8)
    H, I, T = 16, 12, 9
    x = torch.from_numpy(r.standard_normal((T, H)))
    w1, w3 = torch.from_numpy(r.standard_normal((I, H))), torch.from_numpy(r.standard_normal((I, H)))
    w2 = torch.from_numpy(r.standard_normal((H, I)))
    want = torch.nn.functional.linear(
        torch.nn.functional.silu(torch.nn.functional.linear(x, w1)) * torch.nn.functional.linear(x, w3), w2)
    _, y = oracle.grouped_gemm(x.numpy(), np.array([0, T]), w1.numpy()[None], w3.numpy()[None],
                               w2.numpy()[None])
    assert np.allclose(y, want.numpy(), rtol=1e-12, atol=1e-12)


def test_grouped_gemm_skips_empty_blocks():
    r = rng(9)
    E, H, I = 3, 4, 2
    w1, w3, w2 = r.standard_normal((E, I, H)), r.standard_normal((E, I, H)), r.standard_normal((E, H, I))
    w1[1] = w3[1] = np.nan
    w2[1] = np.nan          # expert 1 has no rows: its weights must never be read
    xp = r.standard_normal((3, H))
    _, y = oracle.grouped_gemm(xp, np.array([0, 2, 2, 3]), w1, w3, w2)
    assert np.isfinite(y).all()


# ---------------------------------------------------------------- unpermute

def test_unpermute_identity_experts_k1_is_exact():
    x = rng(10).standard_normal((7, 5))
    ids = synth.random_ids(7, 1, 4, seed=3)
    _, r2f, f2r = oracle.permute(ids, 4)
    xp = oracle.gather_rows(x, r2f, 1)
    out = oracle.unpermute(xp, f2r, np.ones((7, 1)), 7, 1)
    assert np.array_equal(out, x)


def test_unpermute_identity_experts_weights_sum_to_one():
    T, K, E = 11, 3, 6
    x = rng(11).standard_normal((T, 8))
    ids = synth.random_ids(T, K, E, seed=4)
    _, r2f, f2r = oracle.permute(ids, E)
    xp = oracle.gather_rows(x, r2f, K)
    w = rng(12).random((T, K))
    w /= w.sum(1, keepdims=True)
    assert np.allclose(oracle.unpermute(xp, f2r, w, T, K), x, rtol=0, atol=1e-14)


def test_unpermute_adds_gated_shared_expert():
    T, K, H = 3, 2, 4
    y = np.ones((T * K, H))
    f2r = np.arange(T * K)
    w = np.full((T, K), 0.5)
    sh = np.full((T, H), 2.0)
    g = np.array([0.0, 0.5, 1.0])
    out = oracle.unpermute(y, f2r, w, T, K, sh, g)
    assert np.allclose(out, np.array([[1.0] * H, [2.0] * H, [3.0] * H]))


# ---------------------------------------------------------------- whole layer

@pytest.mark.parametrize("mode,shared", [(0, False), (1, False), (0, True)])
def test_layer_matches_brute_force(mode, shared):
    spec = synth.LayerSpec("pin", H=8, E=5, K=2, I=6, mode=mode,
                           routed_scale=2.5 if mode else 1.0, has_shared=shared,
                           I_shared=4 if shared else 0, sel_bias_var=0.1 if mode else 0.0)
    inp = synth.host_inputs(spec, T=6, seed=13)
    res = oracle.moe_layer_from_inputs(inp)
    x = oracle.bf16_to_f64(inp["x_bits"])
    w1, w3, w2 = (np.stack([b[e] for e in range(spec.E)]) for b in oracle.layer_weights_f64(inp))
    sh = None
    if shared:
        sh = tuple(oracle.bf16_to_f64(inp[k]).tolist() for k in ("sw1_bits", "sw3_bits", "sw2_bits"))
    want = brute.layer(x.tolist(), inp["wg"].astype(np.float64).tolist(), None,
                       w1.tolist(), w3.tolist(), w2.tolist(), spec.E, spec.K, mode, spec.routed_scale,
                       None if inp["sel_bias"] is None else inp["sel_bias"].astype(np.float64).tolist(),
                       sh)
    assert np.allclose(res["out"], np.array(want), rtol=1e-6, atol=1e-9)


def test_layer_fp8_equals_bf16_path_on_dequantised_weights():
    spec = synth.LayerSpec("pin8", H=160, E=3, K=2, I=136, wdtype="fp8")
    inp = synth.host_inputs(spec, T=5, seed=14)
    res = oracle.moe_layer_from_inputs(inp)
    w1, w3, w2 = (np.stack([b[e] for e in range(3)]) for b in oracle.layer_weights_f64(inp))
    res2 = oracle.moe_layer(oracle.bf16_to_f64(inp["x_bits"]), inp["wg"], None, None, w1, w3, w2,
                            E=3, K=2, mode=0)
    assert np.array_equal(res["out"], res2["out"])
    # the dequantised weights are the e4m3 values times the block scale
    assert w1[0, 0, 0] == oracle.e4m3_to_f64(inp["w1_q"][0, 0, 0]) * inp["s1"][0, 0, 0]
    assert w1[2, 135, 159] == oracle.e4m3_to_f64(inp["w1_q"][2, 135, 159]) * inp["s1"][2, 1, 1]


# ---------------------------------------------------------------- MXFP4 storage
def test_e2m1_all_codes_closed_form():
    # E2M1 (OCP Microscaling): sign, 2 exponent bits with bias 1, 1 mantissa
    # bit, exponent field 0 = subnormal m * 0.5
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    packed = np.array([[c | (c << 4) for c in range(16)]], np.uint8)  # each code twice
    d = oracle.dequant_mxfp4(packed, np.array([[127]], np.uint8))[0]
    want = np.array(mags + [-m for m in mags])
    assert np.array_equal(d[0::2], want) and np.array_equal(d[1::2], want)
    assert np.signbit(d[16])  # code 8 is -0


def test_mxfp4_golden_worked_example():
    g = json.load(open(os.path.join(GOLD, "mxfp4_worked.json")))
    d = oracle.dequant_mxfp4(np.array([g["packed"]], np.uint8), np.array([g["scales"]], np.uint8))
    assert np.array_equal(d[0], np.array(g["values"]))


def test_mxfp4_scale_is_a_power_of_two_per_32_elements():
    # every scale byte s multiplies its 32 elements by 2^(s - 127), exactly
    packed = np.full((2, 48), 0x22, np.uint8)     # all elements code 2 = 1.0
    scales = np.array([[0, 1, 254], [127, 130, 100]], np.uint8)
    d = oracle.dequant_mxfp4(packed, scales)
    for r in range(2):
        for b in range(3):
            assert (d[r, 32 * b:32 * b + 32] == 2.0 ** (int(scales[r, b]) - 127)).all()


def test_mxfp4_quantisation_round_trip_bound():
    # synth's quantiser then the oracle's decode: every element within one
    # spacing of the e2m1 grid at its block's scale (half a spacing, or the
    # clamp of values in (6, 8) x scale to 6 x scale), zeros exact, values on
    # the grid exact
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((8, 256)) * 0.03).astype(np.float32)
    w[0, :32] = 0.0
    q, s = synth.quantize_mxfp4(w)
    d = oracle.dequant_mxfp4(q, s)
    scale = np.repeat(np.exp2(s.astype(np.float64) - 127.0), 32, axis=1)
    assert (np.abs(d - w) <= 2.0 * scale).all()
    assert (d[0, :32] == 0).all()
    # amax / scale lies in [4, 8): the block's largest element reads 4 or 6
    blk = np.abs(d).reshape(8, 8, 32).max(axis=2) / scale.reshape(8, 8, 32)[:, :, 0]
    assert np.isin(blk[1:], [4.0, 6.0]).all()
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -6] + [0] * 22, np.float32)[None] * 2.0 ** -7
    q, s = synth.quantize_mxfp4(grid.astype(np.float32))
    assert np.array_equal(oracle.dequant_mxfp4(q, s), grid)


def test_mxfp4_device_quantiser_matches_host():
    # the torch rule (device draws) gives the host rule's bits
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(4)
    w = (rng.standard_normal((16, 128)) * 0.05).astype(np.float32)
    w[3, 40] = 0.0
    w[5, :32] = 0.0
    q, s = synth.quantize_mxfp4(w)
    qt, st = synth.quantize_mxfp4_torch(torch.from_numpy(w))
    assert np.array_equal(q, qt.numpy()) and np.array_equal(s, st.numpy())


def test_layer_mxfp4_equals_bf16_path_on_dequantised_weights():
    spec = synth.LayerSpec("pin4", H=160, E=3, K=2, I=96, wdtype="mxfp4")
    inp = synth.host_inputs(spec, T=5, seed=15)
    res = oracle.moe_layer_from_inputs(inp)
    w1, w3, w2 = (np.stack([b[e] for e in range(3)]) for b in oracle.layer_weights_f64(inp))
    assert w1.shape == (3, 96, 160) and w2.shape == (3, 160, 96)
    res2 = oracle.moe_layer(oracle.bf16_to_f64(inp["x_bits"]), inp["wg"], None, None, w1, w3, w2,
                            E=3, K=2, mode=0)
    assert np.array_equal(res["out"], res2["out"])


# ---------------------------------------------------------------- W8A8 activations
def test_e4m3_round_matches_torch_cast():
    # library routine: torch's float32 -> float8_e4m3fn cast rounds to nearest
    # even; compared inside the finite range on every code, every midpoint,
    # the float32 neighbours of every midpoint and random values
    vals = oracle.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2
    m32 = mids.astype(np.float32)
    v = np.concatenate([vals, mids, np.nextafter(m32, np.float32(0)).astype(np.float64),
                        np.nextafter(m32, np.float32(1e9)).astype(np.float64),
                        rng(21).uniform(-448, 448, 4000), rng(22).normal(0, 0.01, 2000)])
    v = np.concatenate([v, -v]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_round(v.astype(np.float64))
    assert np.array_equal(got, ref)


def test_e4m3_round_saturates_and_keeps_sign():
    got = oracle.e4m3_round(np.array([448.0, 449.0, 464.0, 1e6, 3e38, -500.0, -0.0, -1e-9]))
    assert got.tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x80, 0x80]


def test_quantize_act_fp8_closed_forms():
    a = np.zeros((3, 200), np.float32)
    a[0, :128] = oracle.e4m3_to_f64(np.arange(128, dtype=np.uint8) % 0x7F)  # amax 448: s = 1
    a[0, 128:] = -7.0                                                      # narrow last block
    a[1, 5] = 3.0                                                          # one non-zero
    codes, s = oracle.quantize_act_fp8(a)
    assert s.shape == (3, 2) and s.dtype == np.float32
    assert s[0, 0] == 1.0 and np.array_equal(codes[0, :128], np.arange(128) % 0x7F)
    assert s[0, 1] == np.float32(7.0) / np.float32(448.0) and (codes[0, 128:] == 0xFE).all()
    assert s[1, 0] == np.float32(3.0) / np.float32(448.0) and codes[1, 5] == 0x7E
    assert (codes[1, :5] == 0).all() and s[1, 1] == 0 and s[2, 0] == 0 and (codes[2] == 0).all()


def test_quantize_act_fp8_round_trip_bound():
    # each value within half an e4m3 spacing of its block's grid: 2^-4
    # relative for normal codes, 2^-10 * s below the smallest normal
    a = rng(23).normal(0, 1, (6, 300)).astype(np.float32) * rng(24).uniform(0.01, 50, (6, 1))
    codes, s = oracle.quantize_act_fp8(a)
    d = oracle.dequant_act_fp8(codes, s)
    sf = np.repeat(s.astype(np.float64), 128, axis=1)[:, :300]
    assert (np.abs(d - a) <= 2.0 ** -4 * np.abs(a) * (1 + 1e-6) + 2.0 ** -10 * sf).all()
    # the block maximum is always the largest code
    for r in range(6):
        for b in range(3):
            blk = a[r, 128 * b:128 * (b + 1)]
            j = 128 * b + int(np.argmax(np.abs(blk)))
            assert codes[r, j] & 0x7F == 0x7E


def test_quantize_act_fp8_matches_brute_force():
    a = rng(25).normal(0, 2, (3, 150)).astype(np.float32)
    a[1, :20] = 0.0
    codes, s = oracle.quantize_act_fp8(a)
    bc, bs = brute.quant_rows(a.astype(np.float64).tolist())
    assert np.array_equal(codes, np.array(bc, np.uint8))
    assert np.array_equal(s, np.array(bs, np.float32))


def test_round_bf16_matches_torch():
    v = np.concatenate([rng(26).normal(0, 3, 3000), [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]])
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).double().numpy()
    assert np.array_equal(oracle.round_bf16(v), ref)


def test_grouped_gemm_w8a8_matches_brute_force():
    r = rng(27)
    E, H, I = 3, 144, 136  # two scale blocks in each GEMM's K, the second narrow
    offsets = np.array([0, 2, 2, 5])
    xp = oracle.bf16_to_f64(synth.f32_to_bf16_bits(r.normal(0, 1, (5, H)).astype(np.float32)))
    w1 = r.normal(0, H ** -0.5, (E, I, H))
    w3 = r.normal(0, H ** -0.5, (E, I, H))
    w2 = r.normal(0, I ** -0.5, (E, H, I))
    h, y = oracle.grouped_gemm_w8a8(xp, offsets, w1, w3, w2)
    bh, by = brute.grouped_gemm_w8a8(xp.tolist(), offsets.tolist(), w1.tolist(), w3.tolist(),
                                      w2.tolist())
    # the two sum the dot products in different orders: a bf16 rounding of
    # hact may land one step apart
    assert (np.abs(h - np.array(bh)) <= 2.0 ** -8 * np.abs(h)).all()
    assert np.allclose(y, np.array(by), rtol=1e-9, atol=1e-12)
    # the quantised path is near the unquantised one (e4m3 keeps 3 mantissa
    # bits), not equal to it
    h0, y0 = oracle.grouped_gemm(xp, offsets, w1, w3, w2)
    err = np.sqrt(np.mean((y - y0) ** 2)) / np.sqrt(np.mean(y0 ** 2))
    assert 1e-3 < err < 0.1


def test_layer_w8a8_uses_the_quantised_experts():
    spec = synth.LayerSpec("pin8a8", H=160, E=3, K=2, I=136, wdtype="fp8", act="fp8")
    inp = synth.host_inputs(spec, T=5, seed=16)
    res = oracle.moe_layer_from_inputs(inp)
    w1, w3, w2 = (np.stack([b[e] for e in range(3)]) for b in oracle.layer_weights_f64(inp))
    h, y = oracle.grouped_gemm_w8a8(res["xp"], res["offsets"], w1, w3, w2)
    assert np.array_equal(res["y"], y) and np.array_equal(res["hact"], h)
    out = oracle.unpermute(y, res["flat_to_row"], res["weights"], 5, 2)
    assert np.array_equal(res["out"], out)
