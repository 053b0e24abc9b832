"""Full-size workloads (weights drawn on the device), in the launch
configuration the benchmark times: the whole layer through ``moe_layer``.

The oracle recomputes a sample of tokens one by one (routing per token is
independent, so the oracle's layer on the sampled rows gives exactly those
rows), pulling only the experts those tokens use from the device.  Every token
is also checked against properties that hold at any size: distinct experts
per token, weights summing to 1 (or to the routed scale), offsets equal to the
histogram's prefix sum, and a bijective permutation."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_07_gb300 import synth
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mixture_experts_layer_07_gb300 import build
    build.build()
    from mixture_experts_layer_07_gb300 import ops as o
    return o


class DeviceBank:
    """[E, rows, cols] expert weights on the device, fetched per expert."""

    def __init__(self, t, s=None):
        self.t, self.s, self.shape = t, s, tuple(t.shape)

    def __getitem__(self, e):
        if self.s is None:
            return self.t[e].double().cpu().numpy()
        return oracle.dequant_fp8_block(self.t[e].cpu().numpy(), self.s[e].cpu().numpy())


FULL = [("qwen3_30b_a3b", {}, 2048), ("high_expert", {}, 512), ("gpt_oss_20b", {}, 4096),
        ("shared_gate", {}, 1024), ("qwen3_30b_a3b", {}, 1)]


@pytest.mark.parametrize("name,over,T", FULL)
def test_layer_full_size_sampled(ops, name, over, T):
    spec = synth.SPECS[name].with_(**over)
    d = synth.device_inputs(spec, T, seed=5)
    t = {"x": d["x"], "wg": d["wg"], "gate_bias": d["gate_bias"], "sel_bias": d["sel_bias"]}
    if spec.wdtype == "fp8":
        t.update(w1=d["w1_q"], w3=d["w3_q"], w2=d["w2_q"], s1=d["s1"], s3=d["s3"], s2=d["s2"])
    else:
        t.update(w1=d["w1"], w3=d["w3"], w2=d["w2"])
    if spec.has_shared:
        t.update(sw1=d["sw1"], sw3=d["sw3"], sw2=d["sw2"])
    layer = ops.MoELayer(U.config_for(ops, spec, T_max=T), t)
    out = layer(d["x"])
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    E, K = spec.E, spec.K
    ids = layer.view("ids", torch.int32, (T, K)).cpu().numpy()
    w = layer.view("weights", torch.float32, (T, K)).cpu().numpy().astype(np.float64)
    off = layer.view("offsets", torch.int32, (E + 1,)).cpu().numpy()
    r2f = layer.view("row_to_flat", torch.int32, (T * K,)).cpu().numpy()
    f2r = layer.view("flat_to_row", torch.int32, (T * K,)).cpu().numpy()
    # properties over every token
    assert all(len(set(r)) == K for r in ids)
    assert ids.min() >= 0 and ids.max() < E
    target = spec.routed_scale if spec.mode == 1 else 1.0
    assert np.allclose(w.sum(1), target, rtol=1e-5)
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(ids.ravel(), minlength=E))]))
    assert np.array_equal(np.sort(r2f), np.arange(T * K)) and np.array_equal(f2r[r2f], np.arange(T * K))
    o64 = U.f64(out)
    assert np.isfinite(o64).all()
    # sampled tokens through the oracle
    rng = np.random.default_rng(T)
    sample = sorted(set([0, T - 1] + rng.choice(T, size=min(T, 4), replace=False).tolist()))
    xs = d["x"][sample].double().cpu().numpy()
    wg = d["wg"].double().cpu().numpy()
    gb = None if d["gate_bias"] is None else d["gate_bias"].double().cpu().numpy()
    sb = None if d["sel_bias"] is None else d["sel_bias"].cpu().numpy()
    if spec.wdtype == "fp8":
        banks = (DeviceBank(d["w1_q"], d["s1"]), DeviceBank(d["w3_q"], d["s3"]),
                 DeviceBank(d["w2_q"], d["s2"]))
    else:
        banks = (DeviceBank(d["w1"]), DeviceBank(d["w3"]), DeviceBank(d["w2"]))
    shared = None
    if spec.has_shared:
        shared = tuple(d[k].double().cpu().numpy() for k in ("sw1", "sw3", "sw2"))
    res = oracle.moe_layer(xs, wg, gb, sb, *banks, E=E, K=K, mode=spec.mode,
                           routed_scale=spec.routed_scale, shared=shared)
    # tokens whose K-th and (K+1)-th keys nearly tie may route either way
    lg = res["logits"]
    if spec.mode == 0:
        keys = lg[:, :E]
    else:
        keys = oracle.sigmoid_f32(lg.astype(np.float32)[:, :E]).astype(np.float64) + sb[None, :]
    srt = -np.sort(-keys, axis=1)
    clear = (srt[:, K - 1] - srt[:, K]) > 1e-4
    assert np.array_equal(ids[sample][clear], res["ids"][clear])
    rel = 5e-2 if spec.wdtype == "fp8" else 2e-2
    U.assert_bf16_close(o64[sample][clear], res["out"][clear], rel, f"{name} T={T} sampled rows")
