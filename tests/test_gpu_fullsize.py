"""Full-size workloads (weights drawn on the device), in the launch
configuration the benchmark times: the whole layer through ``moe_layer``.

For every full-size layer:

* routing of EVERY token, bit for bit: the oracle's top-K of the GPU's own
  logits gives the same ids (and weights within 1e-5), the oracle's stable
  permute of those ids the same offsets and permutations, and every block's
  variant is the host predicate of its m_size;
* the router logits of sampled tokens against the float64 oracle;
* whole expert blocks, element by element: the hottest and the coldest
  non-empty expert and two more at random -- every hact and y row of each
  block (so every token tile and every 128-feature block of those units)
  against the oracle's expert MLP on the same token rows;
* the layer output of sampled tokens (at least 64 where T allows), with the
  oracle routing the GPU's own logits, so that no near-tied token is left out;
* the shared expert's output of sampled tokens (shared-gate layer).

The oracle pulls only the experts it needs from the device, one at a time."""
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
    """[E, rows, cols] expert weights on the device, fetched per expert and
    widened to float64 exactly (bf16 on the device; e4m3 and e2m1 codes
    dequantised by the oracle on the host)."""

    def __init__(self, t, s=None, fmt="bf16"):
        self.t, self.s, self.fmt = t, s, fmt
        self.shape = tuple(t.shape[:2]) + (t.shape[2] * (2 if fmt == "mxfp4" else 1),)

    def __getitem__(self, e):
        if self.s is None:
            return self.t[e].double().cpu().numpy()
        if self.fmt == "mxfp4":
            return oracle.dequant_mxfp4(self.t[e].cpu().numpy(), self.s[e].cpu().numpy())
        return oracle.dequant_fp8_block(self.t[e].cpu().numpy(), self.s[e].cpu().numpy())

    def __len__(self):
        return self.shape[0]


# (workload, overrides, T, output tokens compared)
FULL = [("qwen3_30b_a3b", {}, 2048, 64), ("qwen3_30b_a3b", {}, 1, 1),
        ("qwen3_30b_a3b", {}, 8, 8),
        ("gpt_oss_20b", {}, 4096, 64), ("gpt_oss_20b", {}, 512, 64), ("gpt_oss_20b", {}, 32, 32),
        ("gpt_oss_20b", {"wdtype": "mxfp4"}, 4096, 64), ("gpt_oss_20b", {"wdtype": "mxfp4"}, 1, 1),
        ("gpt_oss_20b", {"act": "fp8"}, 4096, 64),
        ("shared_gate", {}, 1024, 64), ("shared_gate", {}, 1, 1),
        ("high_expert", {}, 512, 16), ("high_expert", {"E": 512, "K": 16}, 512, 16),
        ("high_expert", {"E": 1024, "K": 9}, 512, 16)]


def sample_tokens(T, n, seed):
    if n >= T:
        return list(range(T))
    rng = np.random.default_rng(seed)
    return sorted(set([0, T - 1] + rng.choice(T, size=n - 2, replace=False).tolist()))


@pytest.mark.parametrize("name,over,T,n_out", FULL,
                         ids=lambda v: ",".join(f"{k}={x}" for k, x in v.items()) or "base"
                         if isinstance(v, dict) else None)
def test_layer_full_size(ops, name, over, T, n_out):
    torch.cuda.empty_cache()
    spec = synth.SPECS[name].with_(**over)
    d = synth.device_inputs(spec, T, seed=5)
    t = {"x": d["x"], "wg": d["wg"], "gate_bias": d["gate_bias"], "sel_bias": d["sel_bias"]}
    fp8 = spec.wdtype == "fp8"
    sfx = {"fp8": "_q", "mxfp4": "_q4"}.get(spec.wdtype)
    if sfx:
        t.update(w1=d["w1" + sfx], w3=d["w3" + sfx], w2=d["w2" + sfx], s1=d["s1"], s3=d["s3"],
                 s2=d["s2"])
    else:
        t.update(w1=d["w1"], w3=d["w3"], w2=d["w2"])
    if spec.has_shared:
        t.update(sw1=d["sw1"], sw3=d["sw3"], sw2=d["sw2"])
    layer = ops.MoELayer(U.config_for(ops, spec, T_max=T), t)
    out = layer(d["x"])
    torch.cuda.synchronize()
    assert int(layer.dev_status.item()) == 0
    E, K, G, H, I = spec.E, spec.K, spec.G, spec.H, spec.I
    R = T * K
    lg = layer.view("logits", torch.float32, (T, G)).cpu().numpy()
    ids = layer.view("ids", torch.int32, (T, K)).cpu().numpy()
    w = layer.view("weights", torch.float32, (T, K)).cpu().numpy()
    off = layer.view("offsets", torch.int32, (E + 1,)).cpu().numpy()
    r2f = layer.view("row_to_flat", torch.int32, (R,)).cpu().numpy()
    f2r = layer.view("flat_to_row", torch.int32, (R,)).cpu().numpy()
    hact = layer.view("hact", torch.bfloat16, (R, I))
    y = layer.view("y", torch.bfloat16, (R, H))
    x64 = U.f64(d["x"])
    wg = d["wg"].double().cpu().numpy()
    gb = None if d["gate_bias"] is None else d["gate_bias"].double().cpu().numpy()
    sb = None if d["sel_bias"] is None else d["sel_bias"].cpu().numpy()

    # routing of every token on the GPU's own logits, bit for bit
    if spec.mode == 0:
        rid, rw = oracle.topk_softmax_renorm(lg.astype(np.float64), E, K)
    else:
        rid, rw = oracle.topk_sigmoid_bias(lg, sb, E, K, spec.routed_scale)
    assert np.array_equal(ids, rid)
    U.assert_weights_close(w, rw)
    if spec.has_shared:
        U.assert_weights_close(layer.view("shared_gate", torch.float32, (T,)).cpu().numpy(),
                               oracle.shared_gate(lg.astype(np.float64), E))
    o_off, o_r2f, o_f2r = oracle.permute(ids, E)
    assert np.array_equal(off, o_off)
    assert np.array_equal(r2f, o_r2f) and np.array_equal(f2r, o_f2r)
    wd = U.wdtype_of(ops, spec)
    want = [ops.block_variant(int(m), R, E, -1, 0, wd) for m in np.diff(off)]
    assert layer.view("block_variant", torch.int32, (E,)).cpu().numpy().tolist() == want

    # router logits of sampled tokens against the float64 oracle
    rs = sample_tokens(T, 64, T + 1)
    U.assert_router_close(lg[rs].astype(np.float64), x64[rs], wg, gb)

    if sfx:
        banks = tuple(DeviceBank(d[k + sfx], d[s], spec.wdtype)
                      for k, s in (("w1", "s1"), ("w3", "s3"), ("w2", "s2")))
    else:
        banks = (DeviceBank(d["w1"]), DeviceBank(d["w3"]), DeviceBank(d["w2"]))
    rel = 5e-2 if fp8 else 2e-2

    # whole expert blocks: hottest, coldest non-empty, two more at random
    m = np.diff(off)
    nz = np.flatnonzero(m)
    pick = list(dict.fromkeys([int(nz[np.argmax(m[nz])]), int(nz[np.argmin(m[nz])])]))
    rng = np.random.default_rng(E + T)
    rest = [int(e) for e in nz if int(e) not in pick]
    pick += [int(e) for e in rng.choice(rest, size=min(2, len(rest)), replace=False)]
    for e in pick:
        lo, hi = int(off[e]), int(off[e + 1])
        a = x64[r2f[lo:hi] // K]
        if spec.act == "fp8":  # W8A8: the rows are quantised one by one
            h_ref, y_ref = oracle.grouped_gemm_w8a8(a, np.array([0, hi - lo]), banks[0][e][None],
                                                    banks[1][e][None], banks[2][e][None])
        else:
            h_ref, y_ref = oracle.expert_swiglu(a, banks[0][e], banks[1][e], banks[2][e])
        U.assert_bf16_close(U.f64(hact[lo:hi]), h_ref, rel, f"{name} T={T} expert {e} hact")
        U.assert_bf16_close(U.f64(y[lo:hi]), y_ref, rel, f"{name} T={T} expert {e} y")

    # the layer output of sampled tokens, routed on the GPU's logits
    sample = sample_tokens(T, n_out, T)
    shared = None
    if spec.has_shared:
        shared = tuple(d[k].double().cpu().numpy() for k in ("sw1", "sw3", "sw2"))
    res = oracle.moe_layer(x64[sample], wg, gb, sb, *banks, E=E, K=K, mode=spec.mode,
                           routed_scale=spec.routed_scale, shared=shared,
                           logits_override=lg[sample].astype(np.float64),
                           w8a8=spec.act == "fp8")
    assert np.array_equal(ids[sample], res["ids"])
    o64 = U.f64(out)
    assert np.isfinite(o64).all()
    U.assert_bf16_close(o64[sample], res["out"], rel, f"{name} T={T} sampled rows")
    if spec.has_shared:
        sh = layer.view("shared_y", torch.bfloat16, (T, H))
        U.assert_bf16_close(U.f64(sh)[sample], res["shared_y"], 2e-2, f"{name} T={T} shared")
    del layer, d, t, banks
    torch.cuda.empty_cache()
