"""The benchmark's roofline accounting on the host: algorithmic bytes and
flops per stage, and which roofline binds.  The grouped GEMM's algorithmic
bytes are checked against the DRAM traffic ncu measured for the same stage
(profiles/traffic.json), so the accounting is tied to a measurement, not only
to its own formula."""
import json
import os

import numpy as np
import pytest

from mixture_experts_layer_07_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    import bench
    return bench


def _peaks():
    b = _bench()
    return {"hbm_gbs": b.FALLBACK_HBM_GBS, "bf16_tflops": b.FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": b.FALLBACK_BF16_TFLOPS, "source": "fallback"}


def test_gemm_bytes_match_measured_dram_traffic():
    # qwen3-30b-a3b T=2048: every expert active; ncu's read + write of the
    # two grouped-GEMM launches at that size is in profiles/traffic.json
    spec = synth.SPECS["qwen3_30b_a3b"]
    st = _bench().stage_bytes_flops(spec, 2048, None, spec.E)
    recs = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))["records"]
    rec = next(r for r in recs if r["workload_name"] == "qwen3_30b_a3b" and r["T"] == 2048)
    measured = rec["traffic_bytes_per_step"]
    assert abs(st["grouped_gemm"]["bytes"] - measured) <= 0.01 * measured


def test_stage_accounting_scales_with_the_batch():
    # doubling T doubles every activation term and leaves the weight terms
    spec = synth.SPECS["qwen3_30b_a3b"]
    b = _bench()
    a1 = b.stage_bytes_flops(spec, 1024, None, spec.E)
    a2 = b.stage_bytes_flops(spec, 2048, None, spec.E)
    H, E, G, I = spec.H, spec.E, spec.G, spec.I
    weights = {"router": 4 * G * H, "grouped_gemm": E * 3 * H * I * 2, "permute": 4 * (E + 1)}
    for k in ("router", "topk", "permute", "grouped_gemm", "unpermute"):
        w = weights.get(k, 0)
        assert a2[k]["bytes"] - w == 2 * (a1[k]["bytes"] - w), k
        assert a2[k]["flops"] == 2 * a1[k]["flops"], k


@pytest.mark.parametrize("name,T,bound", [("qwen3_30b_a3b", 2048, "hbm"),
                                          ("gpt_oss_20b", 4096, "tensor"),
                                          ("shared_gate", 1024, "hbm")])
def test_gemm_roofline_bound(name, T, bound):
    # the ridge: bf16 tensor peak / HBM bandwidth ~ 280 flop per byte; only
    # the FP8 prefill shape with its hot experts is past it
    spec = synth.SPECS[name]
    b = _bench()
    st = b.stage_bytes_flops(spec, T, None, spec.E)["grouped_gemm"]
    r = b.roofline_of(st["bytes"], st["flops"], 1e-3, _peaks(), "tensor")
    assert r["bound"] == bound
    if bound == "hbm":
        assert r["frac"] == pytest.approx(st["bytes"] / 1e-3 / 1e9 / b.FALLBACK_HBM_GBS)
    else:
        assert r["frac"] == pytest.approx(st["flops"] / 1e-3 / 1e12 / b.FALLBACK_BF16_TFLOPS)


def test_router_roofline_on_three_bf16_mmas():
    # the tensor-core router does three bf16 MMAs per fp32 product: its
    # compute ceiling is a third of the bf16 peak
    b = _bench()
    spec = synth.SPECS["qwen3_30b_a3b"]
    st = b.stage_bytes_flops(spec, 262144, None, spec.E)["router"]
    r = b.roofline_of(st["bytes"], st["flops"], 1e-3, _peaks(), "bf16x3")
    assert r["bound"] == "tensor"
    assert r["peak"] == pytest.approx(b.FALLBACK_BF16_TFLOPS / 3)
    assert np.isclose(r["frac"], st["flops"] / 1e-3 / 1e12 / (b.FALLBACK_BF16_TFLOPS / 3))
