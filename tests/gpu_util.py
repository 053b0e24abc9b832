"""Helpers for the GPU parity tests: move synthetic inputs to the device, read
outputs back, and the tolerances the tests use.

Tolerances (float outputs compared element by element with the float64
oracle):
* router logits: |gpu - oracle| <= 1e-5 * sum_h |x_h * w_h| + 1e-6, i.e. relative
  to the natural scale of each dot product (an fp32 sum of H products errs by
  at most ~H * 2^-24 of that scale, far inside 1e-5 for H <= 7168);
* routing weights and the shared gate: 1e-5 relative + 1e-7 absolute;
* bf16 outputs (expert activations, expert outputs, the layer output):
  |gpu - oracle| <= 2e-2 * |oracle| + 2e-2 * rms(oracle) per tensor (5e-2 when
  the expert weights are FP8).  With MXFP4 weights the oracle dequantises the
  same codes exactly, so the bf16 bound of unquantised weights applies.  Each bf16 rounding is 2^-9 relative; the GPU
  path rounds h, y and out once each and accumulates in fp32.
Integer outputs (ids, offsets, permutations) are compared bit for bit.
"""
import numpy as np
import torch

import oracle


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().double().cpu().numpy()


def dev(a, dtype=None):
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def _experts_dev(a, experts, dtype=None):
    """Full-size device tensor holding only the listed experts' slices (the
    other experts' weights are never read by a correct kernel; they are zero)."""
    if experts is None or len(experts) == a.shape[0]:
        return dev(a, dtype)
    t = torch.zeros(a.shape, dtype=dtype or torch.from_numpy(a[:1]).dtype, device="cuda")
    for e in experts:
        src = torch.from_numpy(np.ascontiguousarray(a[e]))
        t[e] = (src.to(dtype) if dtype is not None else src).cuda()
    return t


def _bf16_experts_dev(bits, experts):
    return _experts_dev(np.ascontiguousarray(bits).view(np.int16), experts).view(torch.bfloat16)


def layer_tensors(inp: dict, experts=None) -> dict:
    """Device tensors of a host input dict, under the names MoELayer expects.
    ``experts``: copy only these experts' weights (the rest stay zero)."""
    d = {"x": bf16_dev(inp["x_bits"]), "wg": dev(inp["wg"]), "gate_bias": dev(inp["gate_bias"]),
         "sel_bias": dev(inp["sel_bias"])}
    if "w1_bits" in inp:
        for k in ("w1", "w3", "w2"):
            d[k] = _bf16_experts_dev(inp[k + "_bits"], experts)
    elif "w1_q" in inp or "w1_q4" in inp:
        sfx = "_q" if "w1_q" in inp else "_q4"
        for k, s in (("w1", "s1"), ("w3", "s3"), ("w2", "s2")):
            d[k] = _experts_dev(inp[k + sfx], experts)
            d[s] = dev(inp[s])
    if "sw1_bits" in inp:
        for k in ("sw1", "sw3", "sw2"):
            d[k] = bf16_dev(inp[k + "_bits"])
    return d


def config_for(ops, spec, T_max, **kw):
    return ops.make_config(T_max, spec.H, spec.E, spec.K, spec.I, has_shared=spec.has_shared,
                           I_shared=spec.I_shared, mode=spec.mode, routed_scale=spec.routed_scale,
                           wdtype=wdtype_of(ops, spec), **kw)


def wdtype_of(ops, spec):
    if spec.act == "fp8":
        assert spec.wdtype == "fp8", "W8A8 takes FP8 weights"
        return ops.W8A8_FP8
    return {"bf16": ops.W_BF16, "fp8": ops.W_FP8, "mxfp4": ops.W_MXFP4}[spec.wdtype]


def assert_router_close(gpu, x, wg, bias=None):
    ref = oracle.router_logits(x, wg, bias)
    scale = np.abs(x) @ np.abs(np.asarray(wg, np.float64)).T
    err = np.abs(gpu - ref)
    bound = 1e-5 * scale + 1e-6
    bad = err > bound
    assert not bad.any(), f"{bad.sum()} logits out of tolerance, worst {(err / bound).max():.3g}x"


def assert_bf16_close(gpu, ref, rel=2e-2, what="output"):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    err = np.abs(gpu - ref)
    bound = rel * np.abs(ref) + rel * rms
    bad = err > bound
    assert np.isfinite(gpu).all(), f"{what}: non-finite values"
    assert not bad.any(), (f"{what}: {bad.sum()}/{bad.size} out of tolerance; worst "
                           f"{(err / np.maximum(bound, 1e-30)).max():.3g}x of bound, rms {rms:.3g}")


def assert_weights_close(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref)
    assert (err <= 1e-5 * np.abs(ref) + 1e-7).all(), f"worst {err.max():.3g}"


