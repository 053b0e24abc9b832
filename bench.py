#!/usr/bin/env python
"""Benchmark of the MoE-layer hot path on GB300.

One step = one full layer (router GEMM -> top-K -> permute -> grouped SwiGLU
expert GEMM -> weighted combine) over one batch of T tokens, through
``moe_layer``.  Default workload: the Qwen3-30B-A3B-shaped layer (H=2048,
E=128, K=8, I=768, bf16 experts, softmax top-8 renormalised) at T=2048 tokens,
synthetic inputs drawn on the device.  Expert weights are 1.2 GB, so every
step reads inputs larger than L2 (no flush needed).

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores instead (a bounded token sample per step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload qwen3_30b_a3b] [--T 2048] [--no-sweep]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# FP32 FMA peak from unit counts and clock: 152 SMs x 128 FP32 lanes x 2 flop x 2.07 GHz
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
METRIC = "MoE-layer tokens/s (and us/layer) vs T; per-stage fraction of HBM/tensor roofline"


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------ peaks
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            flat = {}

            def walk(o, pre=""):
                if isinstance(o, dict):
                    for k, v in o.items():
                        walk(v, f"{pre}{k}.")
                else:
                    flat[pre[:-1]] = o
            walk(d)
            hbm = next((v for k, v in flat.items() if k.endswith("hbm_gbs")), None)
            bf = next((v for k, v in flat.items() if k.endswith("bf16_tflops")), None)
            bfs = next((v for k, v in flat.items() if k.endswith("bf16_tflops_sustained")), None)
            if hbm and bf:
                return {"hbm_gbs": float(hbm), "bf16_tflops": float(bf),
                        "bf16_tflops_sustained": float(bfs or bf), "source": "measured"}
        except Exception as e:  # malformed file: fall back, say so
            log("MEASURED_PEAKS.json unreadable:", e)
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ ranks
def max_over_ranks(ms, world, device=None):
    """Slowest rank's time: every rank passes its own, all get the max."""
    if world <= 1:
        return float(ms)
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank_step, steps, world, max_ms):
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time
    (token data-parallel replicas, weak scaling)."""
    return tokens_per_rank_step * steps * world / (max_ms / 1e3)


# ------------------------------------------------------------------ workload
def wd_of(ops, spec):
    if spec.act == "fp8":
        return ops.W8A8_FP8
    return {"bf16": ops.W_BF16, "fp8": ops.W_FP8, "mxfp4": ops.W_MXFP4}[spec.wdtype]


def weight_bytes(spec, n):
    """Stored bytes of n expert-weight elements (MXFP4: half a byte each plus
    one scale byte per 32)."""
    return {"bf16": 2 * n, "fp8": n, "mxfp4": n // 2 + n // 32}[spec.wdtype]


DTYPE_NAME = {"bf16": "bf16", "fp8": "bf16 activations, fp8-e4m3 weights",
              "mxfp4": "bf16 activations, mxfp4 (e2m1 + ue8m0/32) weights"}


def dtype_name(spec):
    if spec.act == "fp8":
        return "fp8-e4m3 weights and expert-GEMM activations (W8A8), bf16 in and out"
    return DTYPE_NAME[spec.wdtype]


def tensors_of(spec, d):
    t = {"x": d["x"], "wg": d["wg"], "gate_bias": d["gate_bias"], "sel_bias": d["sel_bias"]}
    if spec.wdtype in ("fp8", "mxfp4"):
        q = "_q" if spec.wdtype == "fp8" else "_q4"
        t.update(w1=d["w1" + q], w3=d["w3" + q], w2=d["w2" + q], s1=d["s1"], s3=d["s3"],
                 s2=d["s2"])
    else:
        t.update(w1=d["w1"], w3=d["w3"], w2=d["w2"])
    if spec.has_shared:
        t.update(sw1=d["sw1"], sw3=d["sw3"], sw2=d["sw2"])
    return t


def launches_per_layer(spec, T, dispatch=0, m_skinny=16, wide_min=129, num_sms=152):
    """Kernel launches inside one moe_layer call, mirroring the library's
    launch sequence.
      T <= 32: one fused routing launch (router, top-K, permute, GEMM plan);
               with bf16 weights G1 copies its rows from x itself, with FP8
               weights a permute-copy launch follows
      T > 32:  router 1 (2 from T >= 64: weight split + tensor-core GEMM),
               fused routing 1 (top-K, chunk histograms, and in its last CTA
               the scan and the GEMM plan), scatter 1, permute copy 1
      GEMM:    every block skinny (small batch): a G1 and a G2 launch (K
               slices reduced in the kernel); skinny + tile lists: a G1 and a
               G2 launch each running both lists side by side, or one launch
               for everything while the mean rows per expert are <= 64 and
               H <= 3 I (not with the small-batch row gather); with the FP8
               wide list, per list a G1 and a G2 launch (or one fused); 2 on
               the CUDA-core path
      combine 1; a shared expert adds a grouped GEMM with its own plan.
      Small batches under per-block dispatch: T <= 2 (bf16 or W8A16 FP8; MXFP4
      at T = 1): the logits launch (or the fused routing launch), G1 (routing
      the batch in its CTAs where it can) and G2 as CUDA-core matrix-vector
      products (the shared expert inside them) and the combine; bf16 with a
      shared expert at T = 3, 4, or E <= 128 at T = 4..8: the one-launch
      layer.
      W8A8: quantise xp, G1, quantise hact, G2 (every block one kernel)."""
    R = T * spec.K
    if dispatch == 0 and spec.act == "bf16" and (
            (T <= 2 and spec.wdtype in ("bf16", "fp8")) or (T == 1 and spec.wdtype == "mxfp4")):
        return 4
    if (dispatch == 0 and spec.wdtype == "bf16" and spec.act == "bf16" and
            ((spec.has_shared and T <= 4) or (spec.E <= 128 and 4 <= T <= 8))):
        return 1
    if spec.act == "fp8":
        route = 2 if T <= 32 else (2 if T >= ROUTER_TC_MIN_T else 1) + 3
        shared = 3 if spec.has_shared else 0  # its plan, G1, G2 (bf16 shared expert)
        return route + 4 + shared + 1

    def ksplit(units, kdim):
        nk = -(-kdim // 64)
        best, best_cost = 1, None
        for s in range(1, 9):
            kbs = -(-nk // s)
            if s > 1 and kbs < 2:
                break
            cost = -(-(units * s) // num_sms) * (kbs + 2)
            if best_cost is None or cost < best_cost:
                best, best_cost = s, cost
        return best

    def gemm(max_rows, rows, blocks, with_plan, splittable, inter, gather=False):
        n = 1 if with_plan else 0
        if dispatch == 2:
            return n + 2
        tile = max_rows > m_skinny
        wide = spec.wdtype != "bf16" and tile and max_rows >= wide_min
        # tile and wide lists: one G1+G2 launch each (mean rows <= 64, H <= 3 I)
        fused = rows <= 64 * blocks and spec.H <= 3 * inter and not gather
        if splittable and not tile:
            return n + 2  # small batch, all blocks skinny: G1, G2 (K slices reduced in-kernel)
        if tile and not wide:
            return n + (1 if fused else 2)  # both lists side by side in each launch
        n += 2 + (tile + wide) * (1 if fused else 2)
        return n

    if T <= 32:
        gather = spec.wdtype == "bf16"  # bf16: G1 reads its rows from x, no permuted copy
        route = 1 if gather else 2
        g = gemm(T, R, spec.E, with_plan=False, splittable=True, inter=spec.I, gather=gather)
    else:
        route = (2 if T >= ROUTER_TC_MIN_T else 1) + 3  # fused routing, scatter, row copy
        g = gemm(T, R, spec.E, with_plan=False, splittable=False, inter=spec.I)
    shared = (gemm(T, T, 1, with_plan=True, splittable=False, inter=spec.I_shared)
              if spec.has_shared else 0)
    return route + g + shared + 1


def stage_bytes_flops(spec, T, ids, e_active):
    """Algorithmic bytes / flops per stage (each tensor read or written once)."""
    H, E, K, I, G = spec.H, spec.E, spec.K, spec.I, spec.G
    R = T * K
    sb = 0
    if spec.wdtype == "fp8":
        sb = e_active * 4 * 3 * (-(-I // 128)) * (-(-H // 128))
    st = {
        "router": {"bytes": 2 * T * H + 4 * G * H + 4 * T * G, "flops": 2 * T * G * H},
        "topk": {"bytes": 4 * T * G + 8 * T * K + (4 * E if spec.mode == 1 else 0), "flops": 0},
        "permute": {"bytes": 2 * T * H + 2 * R * H + 12 * R + 4 * (E + 1), "flops": 0},
        "grouped_gemm": {"bytes": e_active * weight_bytes(spec, 3 * H * I) + sb + 4 * R * H + 4 * R * I,
                         "flops": 6 * R * H * I},
        "unpermute": {"bytes": 2 * R * H + 2 * T * H + 8 * R + (2 * T * H + 4 * T if spec.has_shared else 0),
                      "flops": 0},
    }
    if spec.has_shared:
        Is = spec.I_shared
        st["grouped_gemm"]["bytes"] += 3 * H * Is * 2 + 4 * T * H + 4 * T * Is
        st["grouped_gemm"]["flops"] += 6 * T * H * Is
    return st


def roofline_of(bytes_, flops, seconds, peaks, compute="tensor", sustained=False):
    """Fraction of the binding roofline: HBM bytes vs. the stage's compute
    ceiling (bf16 tensor cores for the expert GEMM, FP32 FMA pipes for the
    router); whichever takes longer at its peak is the bound."""
    bw = peaks["hbm_gbs"] * 1e9
    if compute == "alu":
        cpk = FP32_ALU_TFLOPS * 1e12
    else:
        cpk = (peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]) * 1e12
        if compute == "bf16x3":  # fp32-accurate GEMM from three bf16 MMAs per product
            cpk /= 3
        if compute == "tensor_fp8":  # e4m3 MMAs: the nominal fp8/bf16 ratio (4.5 / 2.25) x bf16
            cpk *= 2
    t_mem, t_c = bytes_ / bw, flops / cpk
    if t_mem >= t_c:
        ach = bytes_ / seconds / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"]}
    ach = flops / seconds / 1e12
    pk = cpk / 1e12
    bound = "tensor" if compute in ("bf16x3", "tensor") else compute
    return {"bound": bound, "achieved": ach, "peak": pk, "unit": "TFLOP/s", "frac": ach / pk}


STAGE_COMPUTE = {"router": "alu", "topk": "alu", "permute": "alu", "grouped_gemm": "tensor",
                 "unpermute": "alu"}
ROUTER_TC_MIN_T = 64  # the layer's router runs on the tensor cores from this batch size on


def stage_compute(spec, T, n):
    """The compute ceiling a stage is held against."""
    if n == "router":
        return router_compute(T)
    if n == "grouped_gemm" and spec.act == "fp8":
        return "tensor_fp8"
    return STAGE_COMPUTE[n]


def router_compute(T):
    return "bf16x3" if T >= ROUTER_TC_MIN_T else "alu"


def traffic_record(workload, T, kernel_file):
    """Per-launch DRAM traffic of the grouped-GEMM stage for this workload and
    batch from a committed ncu summary (profiles/traffic.json), only while the
    kernel source is unchanged since it was captured; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        rec = json.load(open(p))
        recs = rec.get("records", [rec])
        src = open(os.path.join(ROOT, "mixture_experts_layer_07_gb300", "csrc", kernel_file), "rb").read()
        sha = hashlib.sha256(src).hexdigest()
        for r in recs:
            if (r.get("workload_name") == workload and r.get("T") == T
                    and r.get("source_sha256") == sha):
                return r.get("traffic_bytes_per_step")
        return None
    except Exception:
        return None


# ------------------------------------------------------------------ our arm
# The five workloads, each at the batch its roofline is quoted on: the tiny
# layer, the Qwen3-30B-A3B-shaped layer (the headline line), the GPT-OSS-20B
# shape at its prefill batch (the tensor-bound FP8 case), the 512-expert
# shared-gate layer and the 896-expert routing stress layer.
DEFAULT_CONFIGS = (("tiny", 16), ("qwen3_30b_a3b", 2048), ("gpt_oss_20b", 4096),
                   ("shared_gate", 1024), ("high_expert", 512))
# oracle tokens per CPU-baseline sample (about 5-10 s of host work each)
CPU_TOKENS = {"tiny": 32768, "qwen3_30b_a3b": 32768, "gpt_oss_20b": 4096,
              "shared_gate": 16384, "high_expert": 4}


def make_layer(spec, T, seed, dev):
    from mixture_experts_layer_07_gb300 import ops, synth

    d = synth.device_inputs(spec, T, seed=seed, device=dev)
    t = tensors_of(spec, d)
    cfg = ops.make_config(T, spec.H, spec.E, spec.K, spec.I, has_shared=spec.has_shared,
                          I_shared=spec.I_shared, mode=spec.mode, routed_scale=spec.routed_scale,
                          wdtype=wd_of(ops, spec))
    return d, t, ops.MoELayer(cfg, t, device=dev)


def measure(spec, T, args, rank, world, dev, peaks, light=False):
    """Time one workload at batch T: device-resident steps (the number the
    line reports), the same layer as a CUDA graph, each stage alone against
    its roofline, end to end through host buffers, and (rank 0) a cold-L2 T
    sweep and the oracle on the host cores.  ``light``: N > 1 replicas of a
    secondary workload, steps and stages only."""
    from mixture_experts_layer_07_gb300 import ops

    d, t, layer = make_layer(spec, T, rank, dev)
    x = d["x"]
    out = torch.empty_like(x)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # ---- device-resident timed region.  The clock sampler starts with the
    # warm-up, which runs for at least one second, so its samples cover the GPU
    # under this load right up to and through the timed steps.
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    t_start = time.perf_counter()
    n_w = 0
    while n_w < args.warmup or time.perf_counter() - t_start < 1.0:
        layer(x, out)
        n_w += 1
        if n_w % 50 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        layer(x, out)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    st = int(layer.dev_status.item())
    if st != 0:
        raise RuntimeError(f"{spec.name} T={T}: device status {st}")
    ms_step = ms / args.steps
    tokens = T * args.steps * world

    # ---- the same layer captured once as a CUDA graph and replayed
    graph_ms = None
    if not light:
        try:
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                layer(x, out)
            stream.wait_stream(side)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                layer(x, out)
            for _ in range(args.warmup):
                g.replay()
            torch.cuda.synchronize()
            barrier()
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            for _ in range(args.steps):
                g.replay()
            g1.record(stream)
            torch.cuda.synchronize()
            graph_ms = max_over_ranks(g0.elapsed_time(g1), world, dev)
            del g
        except Exception as e:  # report, do not hide: the stream number stands
            log("graph capture failed:", repr(e))

    # ---- per-stage times (same workspace, stages called one by one)
    L = layer.layout
    ws = layer.workspace
    E, K, H, I, G = spec.E, spec.K, spec.H, spec.I, spec.G
    R = T * K

    def v(name, dtype, shape):
        return layer.view(name, dtype, shape)

    logits = v("logits", torch.float32, (T, G))
    ids = v("ids", torch.int32, (T, K))
    wts = v("weights", torch.float32, (T, K))
    gsh = v("shared_gate", torch.float32, (T,)) if spec.has_shared else None
    off = v("offsets", torch.int32, (E + 1,))
    r2f = v("row_to_flat", torch.int32, (R,))
    f2r = v("flat_to_row", torch.int32, (R,))
    xp = v("xp", torch.bfloat16, (R, H))
    hact = v("hact", torch.bfloat16, (R, I))
    y = v("y", torch.bfloat16, (R, H))
    pscr = ws[L.permute_scratch:L.gemm_scratch]
    gscr = ws[L.gemm_scratch:L.shared_gemm_scratch]
    sh_scr = ws[L.shared_gemm_scratch:L.total]
    sh_h = v("shared_hact", torch.bfloat16, (T, spec.I_shared)) if spec.has_shared else None
    sh_y = v("shared_y", torch.bfloat16, (T, H)) if spec.has_shared else None
    wd = wd_of(ops, spec)
    names = ["router", "topk", "permute", "grouped_gemm", "unpermute"]
    rscr = ws[L.router_split:L.splitk]

    def router():
        if T >= ROUTER_TC_MIN_T:
            ops.router_gemm_tc(x, t["wg"], t["gate_bias"], logits, rscr, layer.dev_status)
        else:
            ops.router_gemm(x, t["wg"], t["gate_bias"], logits)

    def stages():
        yield router
        yield lambda: ops.topk_route(logits, E, K, spec.mode, spec.routed_scale, ids, wts,
                                     t["sel_bias"], gsh)
        yield lambda: ops.permute(x, ids, E, off, r2f, f2r, xp, pscr, layer.dev_status)

        def gg():
            ops.grouped_gemm(xp, off, E, H, I, t["w1"], t["w3"], t["w2"], hact, y, gscr, wdtype=wd,
                             s1=t.get("s1"), s3=t.get("s3"), s2=t.get("s2"),
                             dev_status=layer.dev_status)
            if spec.has_shared:
                ops.grouped_gemm(x, None, 1, H, spec.I_shared, t["sw1"], t["sw3"], t["sw2"], sh_h,
                                 sh_y, sh_scr, dev_status=layer.dev_status)
        yield gg
        yield lambda: ops.unpermute(y, f2r, wts, T, K, H, out, sh_y, gsh)

    n_stage_steps = max(3, min(args.steps, 20))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n_stage_steps)]
    for s in range(n_stage_steps + 2):
        rec = s >= 2
        if rec:
            evs[s - 2][0].record(stream)
        for i, fn in enumerate(stages()):
            fn()
            if rec:
                evs[s - 2][i + 1].record(stream)
    torch.cuda.synchronize()
    stage_ms = {n: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs)
                for i, n in enumerate(names)}
    ids_h = ids.cpu().numpy()
    e_active = int(len(np.unique(ids_h)))
    sbf = stage_bytes_flops(spec, T, ids_h, e_active)
    per_stage = {}
    for n in names:
        kind = stage_compute(spec, T, n)
        r = roofline_of(sbf[n]["bytes"], sbf[n]["flops"], stage_ms[n] / 1e3, peaks, kind)
        per_stage[n] = {"us": round(stage_ms[n] * 1e3, 2), "bound": r["bound"],
                        "frac": round(r["frac"], 4)}
    dom = max(names, key=lambda n: stage_ms[n])
    roof = roofline_of(sbf[dom]["bytes"], sbf[dom]["flops"], stage_ms[dom] / 1e3, peaks,
                       stage_compute(spec, T, dom))
    roof = {k: (round(v, 4) if isinstance(v, float) else v) for k, v in roof.items()}
    roof["kernel"] = dom
    roof["algorithmic"] = ({"bytes": sbf[dom]["bytes"]} if roof["unit"] == "GB/s"
                           else {"flops": sbf[dom]["flops"]})
    roof["peak_source"] = f"of {peaks['source']}"
    roof["traffic"] = (traffic_record(spec.name, T, "grouped_gemm.cu")
                       if dom == "grouped_gemm" else None)
    hot = (float(np.isin(ids_h, list(spec.hot_experts)).mean()) if spec.hot_experts else None)

    res = {"workload": spec.name, "T": T, "H": spec.H, "E": spec.E, "K": spec.K, "I": spec.I,
           "dtype": dtype_name(spec),
           "us_per_layer": round(ms_step * 1e3, 2),
           "tokens_per_s": round(job_throughput(T, args.steps, world, ms), 1),
           "ms_total": ms, "roofline": roof, "per_stage": per_stage, "clocks": clk,
           "e_active": e_active, "gpu_launches_per_layer": launches_per_layer(spec, T)}
    if hot is not None:
        res["hot_expert_share"] = round(hot, 4)
    if graph_ms is not None:
        res["graph"] = {"value": round(tokens / (graph_ms / 1e3), 1), "unit": "tokens/s",
                        "us_per_layer": round(graph_ms / args.steps * 1e3, 2),
                        "note": "same layer captured once as a CUDA graph, replayed K times"}
    if light:
        del layer, d, t
        torch.cuda.empty_cache()
        return res

    # ---- end to end through the C ABI with host buffers.  Every step copies
    # its input from pinned host memory and its output back to pinned host
    # memory.  When a step's copies are large (>= 1 MB each way) they run on
    # their own streams (one per direction) with two device buffers each way,
    # so one step's copies overlap its neighbours' layers, the way a serving
    # loop pipelines them: the input copy of step i waits until layer i-2 is
    # done with that buffer, layer i waits for its input and for the output
    # copy of step i-2, the output copy of step i waits for layer i.  Small
    # copies stay on the layer's stream in order (there the cross-stream
    # waits would cost more than the copies).  The events bracket all K
    # steps, copies included.
    io_bytes = x.numel() * x.element_size()
    pipelined = io_bytes >= (1 << 20)
    h2d_stream, d2h_stream = ((torch.cuda.Stream(), torch.cuda.Stream()) if pipelined
                              else (stream, stream))
    x_host = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    x_host.copy_(x)
    out_host = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for _ in range(2)]
    x_dev = [torch.empty_like(x) for _ in range(2)]
    out_dev = [torch.empty_like(x) for _ in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_steps(n):
        for i in range(n):
            b = i % 2
            if not pipelined:
                x_dev[b].copy_(x_host, non_blocking=True)
                layer(x_dev[b], out_dev[b], stream=stream)
                out_host[b].copy_(out_dev[b], non_blocking=True)
                continue
            h2d_stream.wait_event(ev_done[b])          # layer i-2 read x_dev[b]
            with torch.cuda.stream(h2d_stream):
                x_dev[b].copy_(x_host, non_blocking=True)
            ev_in[b].record(h2d_stream)
            stream.wait_event(ev_in[b])
            stream.wait_event(ev_out[b])               # step i-2's output copied out
            layer(x_dev[b], out_dev[b], stream=stream)
            ev_done[b].record(stream)
            d2h_stream.wait_event(ev_done[b])
            with torch.cuda.stream(d2h_stream):
                out_host[b].copy_(out_dev[b], non_blocking=True)
            ev_out[b].record(d2h_stream)

    e2e_steps(args.warmup)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(h2d_stream)
    e2e_steps(args.steps)
    e1.record(d2h_stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    # every step's output reached the host
    assert torch.equal(out_host[(args.steps - 1) % 2].to(dev), out_dev[(args.steps - 1) % 2])
    res["e2e"] = {"value": round(tokens / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                  "h2d_bytes_per_step": io_bytes, "d2h_bytes_per_step": io_bytes,
                  "note": ("pinned host buffers; copies on their own streams, double-buffered, "
                           "overlapping neighbouring steps' layers") if pipelined else
                          "pinned host buffers; copies in order on the layer's stream"}
    del x_host, out_host, x_dev, out_dev

    # ---- T sweep (rank 0 only, short): stream launches and graph replay.
    # Below T ~ 100 the experts a call touches fit in L2, so every timed call
    # is preceded by a 256 MB write (outside its events) that flushes L2.
    if rank == 0 and args.sweep:
        sweep = []
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

        def cold(fn):
            return cold_us(fn, stream, flush)

        for Ts in spec.T_sweep:
            if Ts > T:
                continue
            xs = x[:Ts]
            os_ = out[:Ts]
            us = cold(lambda: layer(xs, os_))
            row = {"T": Ts, "us_per_layer": round(us, 2), "tokens_per_s": round(Ts / us * 1e6, 1),
                   "l2": "flushed before each call", "stat": "mean of 40 calls, 4 dropped each end"}
            try:
                gs = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gs):
                    layer(xs, os_)
                ug = cold(gs.replay)
                row.update(graph_us_per_layer=round(ug, 2), graph_tokens_per_s=round(Ts / ug * 1e6, 1))
                del gs
            except Exception as e:
                log("graph capture failed:", repr(e))
            sweep.append(row)
        del flush
        res["sweep"] = sweep
        if int(layer.dev_status.item()) != 0:
            raise RuntimeError(f"{spec.name}: device status {int(layer.dev_status.item())}")

    # ---- CPU baseline (rank 0, N=1 only): the oracle on the host cores
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(spec, d, args.cpu_tokens or CPU_TOKENS[spec.name])
    del layer, d, t
    torch.cuda.empty_cache()
    return res


def run_ours(args, rank, world, local_rank):
    from mixture_experts_layer_07_gb300 import synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks = load_peaks()
    head_spec = workload_spec(args)
    head = measure(head_spec, args.T, args, rank, world, dev, peaks)
    spec, T = head_spec, args.T
    res = {
        "metric": METRIC,
        "value": head["tokens_per_s"],
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(head["ms_total"] / args.steps, 4),
        "us_per_layer": head["us_per_layer"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": head["dtype"],
        "data": "synthetic (seeded; random-init weights of the named layer shape)",
        "config": {"workload": f"{spec.name} MoE layer", "T": T, "H": spec.H, "E": spec.E,
                   "K": spec.K, "I": spec.I, "routing": "softmax top-K renormalised"
                   if spec.mode == 0 else "sigmoid+bias top-K, scaled-sum", "tokens_per_gpu": T,
                   "parallelism": f"token-dp replicas x{world}",
                   "l2": "inputs larger than L2 (expert weights "
                         f"{weight_bytes(spec, spec.E * 3 * spec.H * spec.I) / 1e9:.2f} GB "
                         "per layer), no flush"},
        "roofline": head["roofline"],
        "per_stage": head["per_stage"],
        "graph": head.get("graph"),
        "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches_per_layer"] * args.steps,
        "clocks": head["clocks"],
        "cpu_baseline": head.get("cpu_baseline"),
    }
    if "sweep" in head:
        res["sweep"] = head["sweep"]
    if args.configs:
        # every workload at its own batch (the headline's entry is the headline
        # measurement itself); each entry carries its own roofline, per-stage
        # fractions, CPU baseline and T sweep
        confs = []
        for name, Tc in DEFAULT_CONFIGS:
            if name == head_spec.name and Tc == args.T:
                r = head
            else:
                r = measure(synth.SPECS[name], Tc, args, rank, world, dev, peaks,
                            light=world > 1)
            confs.append({k: v for k, v in r.items() if k != "ms_total"})
        res["configs"] = confs
    if rank == 0 and args.extra:
        res["stage_sweep_large_T"] = stage_sweep(synth.SPECS["qwen3_30b_a3b"],
                                                 (16384, 65536, 262144), peaks, dev)
        res["stage_sweep_large_T_high_expert"] = stage_sweep(synth.SPECS["high_expert"],
                                                             (16384,), peaks, dev)
        res["prefill_grouped_gemm"] = prefill_points(peaks, dev)
        res["weight_formats_gpt_oss_20b"] = format_sweep(peaks, dev)
    return res


# ------------------------------------------------------------------ extra sweeps
def _time(fn, n, stream):
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(n):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n / 1e3  # seconds


def stage_sweep(spec, Ts, peaks, dev):
    """R, K, P, U alone at large T (the sizes where their bytes, not launch
    latency, set the time); each against its own roofline."""
    from mixture_experts_layer_07_gb300 import ops, synth

    stream = torch.cuda.current_stream()
    out = []
    H, E, K, G = spec.H, spec.E, spec.K, spec.G
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    wg = (torch.randn(G, H, device=dev, generator=gen) / H ** 0.5).contiguous()
    for T in Ts:
        R = T * K
        x = torch.randn(T, H, device=dev, generator=gen).to(torch.bfloat16)
        logits = torch.empty(T, G, device=dev)
        ids = torch.empty(T, K, dtype=torch.int32, device=dev)
        w = torch.empty(T, K, device=dev)
        off = torch.empty(E + 1, dtype=torch.int32, device=dev)
        r2f = torch.empty(R, dtype=torch.int32, device=dev)
        f2r = torch.empty(R, dtype=torch.int32, device=dev)
        xp = torch.empty(R, H, dtype=torch.bfloat16, device=dev)
        scratch = torch.empty(ops.permute_scratch_bytes(T, E, K), dtype=torch.uint8, device=dev)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        o = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        sel_bias = torch.zeros(E, device=dev) if spec.mode == 1 else None
        sb = stage_bytes_flops(spec, T, None, 0)
        row = {"T": T}
        rscr = torch.empty(ops.router_tc_scratch_bytes(H, G), dtype=torch.uint8, device=dev)
        t = _time(lambda: ops.router_gemm_tc(x, wg, None, logits, rscr, st), 5, stream)
        r = roofline_of(sb["router"]["bytes"], sb["router"]["flops"], t, peaks, "bf16x3")
        row["router"] = {"us": round(t * 1e6, 1), "bound": r["bound"], "frac": round(r["frac"], 3)}
        t = _time(lambda: ops.router_gemm(x, wg, None, logits), 5, stream)
        r = roofline_of(sb["router"]["bytes"], sb["router"]["flops"], t, peaks, "alu")
        row["router_fp32_simt"] = {"us": round(t * 1e6, 1), "bound": r["bound"],
                                   "frac": round(r["frac"], 3)}
        t = _time(lambda: ops.topk_route(logits, E, K, spec.mode, spec.routed_scale, ids, w,
                                         sel_bias), 10, stream)
        r = roofline_of(sb["topk"]["bytes"], 0, t, peaks, "alu")
        row["topk"] = {"us": round(t * 1e6, 1), "GB/s": round(r["achieved"], 1), "frac": round(r["frac"], 3)}
        t = _time(lambda: ops.permute(x, ids, E, off, r2f, f2r, xp, scratch, st), 5, stream)
        r = roofline_of(sb["permute"]["bytes"], 0, t, peaks, "alu")
        row["permute"] = {"us": round(t * 1e6, 1), "GB/s": round(r["achieved"], 1), "frac": round(r["frac"], 3)}
        t = _time(lambda: ops.unpermute(xp, f2r, w, T, K, H, o), 5, stream)
        r = roofline_of(sb["unpermute"]["bytes"], 0, t, peaks, "alu")
        row["unpermute"] = {"us": round(t * 1e6, 1), "GB/s": round(r["achieved"], 1), "frac": round(r["frac"], 3)}
        out.append(row)
        del x, logits, ids, w, off, r2f, f2r, xp, scratch, o, rscr
        torch.cuda.empty_cache()
    return out


def probe_stages(spec, T, reps, dev):
    """R, K, P, U alone at T, `reps` times, no timing: the command the
    per-stage ncu captures profile."""
    from mixture_experts_layer_07_gb300 import ops

    H, E, K, G = spec.H, spec.E, spec.K, spec.G
    gen = torch.Generator(device=dev)
    gen.manual_seed(1)
    x = torch.randn(T, H, device=dev, generator=gen).to(torch.bfloat16)
    wg = torch.randn(G, H, device=dev, generator=gen) / H ** 0.5
    logits = torch.empty(T, G, device=dev)
    ids = torch.empty(T, K, dtype=torch.int32, device=dev)
    w = torch.empty(T, K, device=dev)
    R = T * K
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    r2f = torch.empty(R, dtype=torch.int32, device=dev)
    f2r = torch.empty(R, dtype=torch.int32, device=dev)
    xp = torch.empty(R, H, dtype=torch.bfloat16, device=dev)
    scr = torch.empty(ops.permute_scratch_bytes(T, E, K), dtype=torch.uint8, device=dev)
    o = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    sel_bias = torch.zeros(E, device=dev) if spec.mode == 1 else None
    rscr = torch.empty(ops.router_tc_scratch_bytes(H, G), dtype=torch.uint8, device=dev)
    for _ in range(reps):
        if T >= ROUTER_TC_MIN_T:
            ops.router_gemm_tc(x, wg, None, logits, rscr)
        else:
            ops.router_gemm(x, wg, None, logits)
        ops.topk_route(logits, E, K, spec.mode, spec.routed_scale, ids, w, sel_bias)
        ops.permute(x, ids, E, off, r2f, f2r, xp, scr)
        ops.unpermute(xp, f2r, w, T, K, H, o)
    torch.cuda.synchronize()
    return {"probe": "stages", "workload": spec.name, "T": T, "reps": reps}


def probe_topk(spec, T, reps, dev):
    """moe_topk_route alone at T on seeded random logits of the workload's
    E, K and score mode, `reps` calls, no timing (for ncu captures)."""
    from mixture_experts_layer_07_gb300 import ops

    E, K = spec.E, spec.K
    gen = torch.Generator(device=dev)
    gen.manual_seed(2)
    logits = torch.randn(T, E, device=dev, generator=gen)
    ids = torch.empty(T, K, dtype=torch.int32, device=dev)
    w = torch.empty(T, K, device=dev)
    sel_bias = (torch.randn(E, device=dev, generator=gen) * 0.3) if spec.mode == 1 else None
    for _ in range(reps):
        ops.topk_route(logits, E, K, spec.mode, spec.routed_scale, ids, w, sel_bias)
    torch.cuda.synchronize()
    return {"probe": "topk", "workload": spec.name, "T": T, "reps": reps}


def probe_layer(spec, T, reps, dev):
    """The whole layer (``moe_layer``) at T, `reps` calls, no timing: the
    command the per-kernel ncu captures of the layer profile."""
    from mixture_experts_layer_07_gb300 import ops, synth

    d = synth.device_inputs(spec, T, seed=1, device=dev)
    t = tensors_of(spec, d)
    cfg = ops.make_config(T, spec.H, spec.E, spec.K, spec.I, has_shared=spec.has_shared,
                          I_shared=spec.I_shared, mode=spec.mode, routed_scale=spec.routed_scale,
                          wdtype=wd_of(ops, spec))
    layer = ops.MoELayer(cfg, t, device=dev)
    out = torch.empty_like(d["x"])
    for _ in range(reps):
        layer(d["x"], out)
    torch.cuda.synchronize()
    st = int(layer.dev_status.item())
    if st != 0:
        raise RuntimeError(f"device status {st}")
    return {"probe": "layer", "workload": spec.name, "T": T, "reps": reps}


def prefill_points(peaks, dev):
    """The grouped GEMM stage on prefill shapes where it is tensor-bound."""
    from mixture_experts_layer_07_gb300 import ops, synth

    stream = torch.cuda.current_stream()
    res = []
    for name, T, over in (("qwen3_30b_a3b", 16384, {}), ("gpt_oss_20b", 4096, {}),
                          ("gpt_oss_20b", 4096, {"act": "fp8"})):
        spec = synth.SPECS[name].with_(**over)
        d = synth.device_inputs(spec, T, seed=3, device=dev)
        t = tensors_of(spec, d)
        cfg = ops.make_config(T, spec.H, spec.E, spec.K, spec.I,
                              wdtype=wd_of(ops, spec))
        layer = ops.MoELayer(cfg, t, device=dev)
        layer(d["x"])
        torch.cuda.synchronize()
        E, K, H, I = spec.E, spec.K, spec.H, spec.I
        R = T * K
        off = layer.view("offsets", torch.int32, (E + 1,))
        xp = layer.view("xp", torch.bfloat16, (R, H))
        hact = layer.view("hact", torch.bfloat16, (R, I))
        y = layer.view("y", torch.bfloat16, (R, H))
        L = layer.layout
        gscr = layer.workspace[L.gemm_scratch:L.shared_gemm_scratch]
        wd = wd_of(ops, spec)
        sec = _time(lambda: ops.grouped_gemm(xp, off, E, H, I, t["w1"], t["w3"], t["w2"], hact, y,
                                             gscr, wdtype=wd, s1=t.get("s1"), s3=t.get("s3"),
                                             s2=t.get("s2")), 10, stream)
        ids = layer.view("ids", torch.int32, (T, K)).cpu().numpy()
        e_act = int(len(np.unique(ids)))
        sb = stage_bytes_flops(spec, T, ids, e_act)["grouped_gemm"]
        kind = "tensor_fp8" if spec.act == "fp8" else "tensor"
        r = roofline_of(sb["bytes"], sb["flops"], sec, peaks, kind)
        hot = float(np.isin(ids, list(spec.hot_experts)).mean()) if spec.hot_experts else None
        res.append({"workload": name + (" W8A8" if spec.act == "fp8" else ""), "T": T,
                    "us": round(sec * 1e6, 1), "bound": r["bound"], "peak": round(r["peak"], 1),
                    "achieved": round(r["achieved"], 1), "unit": r["unit"],
                    "frac": round(r["frac"], 3), "tflops": round(sb["flops"] / sec / 1e12, 1),
                    "hot_expert_share": hot})
        del layer, d, t
        torch.cuda.empty_cache()
    return res


def cold_us(fn, stream, flush, n=40):
    """Device time of fn() in us with L2 flushed (a write of `flush`, outside
    the events) before each of n calls: the mean of the middle 80 % (the
    events tick in ~2 us steps on this part; the trimmed mean resolves below
    one tick)."""
    for _ in range(3):
        fn()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for i in range(n):
        flush.fill_(i & 0xFF)
        evs[i][0].record(stream)
        fn()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    ts = sorted(a.elapsed_time(b) for a, b in evs)
    k = len(ts) // 10
    return statistics.mean(ts[k:len(ts) - k]) * 1e3


def format_sweep(peaks, dev, Ts=(1, 32, 512, 4096)):
    """The GPT-OSS-20B-shaped layer with its expert weights stored three ways
    (bf16, FP8 e4m3 + 128x128 scales, MXFP4): device-resident moe_layer time
    and the grouped GEMM's share of the HBM roofline (weight bytes of the
    active experts over the layer time, the bound of small batches)."""
    from mixture_experts_layer_07_gb300 import synth

    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    res = []
    for wdt in ("bf16", "fp8", "mxfp4", "w8a8"):
        spec = synth.SPECS["gpt_oss_20b"].with_(wdtype="fp8" if wdt == "w8a8" else wdt,
                                                act="fp8" if wdt == "w8a8" else "bf16")
        d, t, layer = make_layer(spec, max(Ts), 3, dev)
        for T in Ts:
            x = d["x"][:T].contiguous()
            out = torch.empty_like(x)
            # below T ~ 100 the touched experts fit in L2: flush before each call
            cold = T < 100
            sec = (cold_us(lambda: layer(x, out), stream, flush) * 1e-6 if cold
                   else _time(lambda: layer(x, out), 20, stream))
            if int(layer.dev_status.item()) != 0:
                raise RuntimeError(f"device status {int(layer.dev_status.item())}")
            ids = layer.view("ids", torch.int32, (T, spec.K)).cpu().numpy()
            e_act = int(len(np.unique(ids)))
            wbytes = e_act * weight_bytes(spec, 3 * spec.H * spec.I)
            res.append({"weights": wdt, "T": T, "us_per_layer": round(sec * 1e6, 2),
                        "tokens_per_s": round(T / sec, 1), "e_active": e_act,
                        "weight_GB_per_s": round(wbytes / sec / 1e9, 1),
                        "weight_frac_of_hbm": round(wbytes / sec / 1e9 / peaks["hbm_gbs"], 3),
                        "l2": "flushed before each call" if cold else "streamed (inputs > L2)"})
        del layer, d, t
        torch.cuda.empty_cache()
    del flush
    return res


# ------------------------------------------------------------------ oracle arm
def host_workload(spec, T, seed=0):
    """The workload drawn on the host (tokens + every expert's weights)."""
    from mixture_experts_layer_07_gb300 import synth
    return synth.host_inputs(spec, T, seed=seed)


def oracle_time(inp, t0, n):
    """Seconds the CPU oracle takes for tokens [t0, t0 + n) of ``inp``."""
    import oracle
    sub = dict(inp)
    sub["x_bits"] = inp["x_bits"][t0:t0 + n]
    sub["T"] = n
    start = time.perf_counter()
    oracle.moe_layer_from_inputs(sub)
    return time.perf_counter() - start


class HostExperts:
    """[E, rows, cols] stored expert weights on the host, holding only the
    experts a sample of tokens routes to (indexing another one is an error)."""

    def __init__(self, shape, parts):
        self.shape, self.parts = tuple(shape), parts

    def __getitem__(self, e):
        return self.parts[int(e)]

    def __len__(self):
        return self.shape[0]


def oracle_inputs_from_device(spec, d, tokens, seed=0):
    """An oracle input dict for `tokens` host-drawn tokens of the workload,
    with the gate and the expert weights copied from the device draw ``d``:
    only the experts the oracle's own routing of those tokens picks (found
    before any timing), so a layer with tens of GB of experts needs only
    what the sample touches on the host."""
    import oracle
    from mixture_experts_layer_07_gb300 import synth

    inp = synth.host_inputs(spec, tokens, seed=seed, weights=False)
    inp["wg"] = d["wg"].cpu().numpy()
    inp["gate_bias"] = None if d["gate_bias"] is None else d["gate_bias"].cpu().numpy()
    inp["sel_bias"] = None if d["sel_bias"] is None else d["sel_bias"].cpu().numpy()
    x = oracle.bf16_to_f64(inp["x_bits"])
    lg = oracle.router_logits(x, inp["wg"], inp["gate_bias"])
    if spec.mode == 0:
        ids, _ = oracle.topk_softmax_renorm(lg, spec.E, spec.K)
    else:
        ids, _ = oracle.topk_sigmoid_bias(lg.astype(np.float32), inp["sel_bias"], spec.E,
                                          spec.K, spec.routed_scale)
    used = sorted(set(ids.ravel().tolist()))

    def bits(t):
        return t.view(torch.int16).cpu().numpy().view(np.uint16)

    if spec.wdtype in ("fp8", "mxfp4"):
        sfx = "_q" if spec.wdtype == "fp8" else "_q4"
        for k, sk in (("w1", "s1"), ("w3", "s3"), ("w2", "s2")):
            q, s = d[k + sfx], d[sk]
            inp[k + sfx] = HostExperts(q.shape, {e: q[e].cpu().numpy() for e in used})
            inp[sk] = HostExperts(s.shape, {e: s[e].cpu().numpy() for e in used})
    else:
        for k in ("w1", "w3", "w2"):
            w = d[k]
            inp[k + "_bits"] = HostExperts(w.shape, {e: bits(w[e]) for e in used})
    if spec.has_shared:
        for k in ("sw1", "sw3", "sw2"):
            inp[k + "_bits"] = bits(d[k])
    return inp, len(used)


def cpu_baseline(spec, d, tokens):
    """The oracle as it stands, timed on the host cores on a bounded sample of
    the workload (`tokens` tokens, the experts they route to)."""
    cores = len(os.sched_getaffinity(0))
    inp, n_exp = oracle_inputs_from_device(spec, d, tokens)
    sec = oracle_time(inp, 0, tokens)
    return {"value": round(tokens / sec, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{tokens} tokens of the {spec.name} workload (same shapes; gate and the "
                      f"{n_exp} experts they route to copied from the device draw), float64 "
                      f"numpy oracle, one pass, {sec:.1f} s"}


def run_reference(args):
    spec = workload_spec(args)
    cores = len(os.sched_getaffinity(0))
    n = max(1, args.ref_tokens)
    inp = host_workload(spec, n * (args.steps + args.warmup), seed=1)
    for w in range(args.warmup):
        oracle_time(inp, w * n, n)
    total = 0.0
    for s in range(args.steps):
        total += oracle_time(inp, (args.warmup + s) * n, n)
    tokens = n * args.steps
    val = tokens / total
    sample = (f"{n} tokens per step of the {spec.name} workload (T={args.T} batch shape, all "
              f"{spec.E} experts), float64 numpy oracle on the host cores")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(val, 3),
        "unit": "tokens/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": f"{spec.name} MoE layer", "T": args.T, "H": spec.H, "E": spec.E,
                   "K": spec.K, "I": spec.I},
        "cpu_baseline": {"value": round(val, 3), "unit": "tokens/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(val, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def _free_port():
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def spawn_ranks(n):
    """Run this script as n ranks on this node and return their exit status."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def print_launch_check(rank, world):
    """Rank start-up and the timing reduction alone, on CPU over gloo: every
    rank reports a time of its own, the slowest one wins, rank 0 prints it."""
    if world > 1:
        torch.distributed.init_process_group("gloo")
    try:
        ms = max_over_ranks(10.0 + rank, world)
        if rank == 0:
            print(json.dumps({"launch_check": True, "n_gpus": world, "max_ms": ms,
                              "value": job_throughput(1, 1, world, ms)}), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


def workload_spec(args):
    """The named workload, with --act applied (fp8: W8A8 on fp8 weights)."""
    from mixture_experts_layer_07_gb300 import synth

    spec = synth.SPECS[args.workload]
    if args.wdtype:
        spec = spec.with_(wdtype=args.wdtype)
    if args.act == "fp8":
        spec = spec.with_(wdtype="fp8", act="fp8")
    elif args.act == "bf16":
        spec = spec.with_(act="bf16")
    return spec


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen3_30b_a3b")
    ap.add_argument("--wdtype", default=None, choices=["bf16", "fp8", "mxfp4"],
                    help="expert weight format of the probed workload")
    ap.add_argument("--act", default=None, choices=["bf16", "fp8"],
                    help="expert-GEMM activations of the probed workload (fp8: W8A8, fp8 weights)")
    ap.add_argument("--T", type=int, default=2048)
    ap.add_argument("--cpu-tokens", type=int, default=0,
                    help="oracle tokens per CPU-baseline sample (0: per-workload default)")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="time only the headline workload, not all five")
    ap.add_argument("--no-extra", dest="extra", action="store_false",
                    help="skip the large-T stage sweep and the prefill GEMM points")
    ap.add_argument("--launch-check", action="store_true",
                    help="rank start-up and max-over-ranks timing only, on CPU (gloo)")
    ap.add_argument("--ref-tokens", type=int, default=256)
    ap.add_argument("--no-sweep", dest="sweep", action="store_false")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--probe-stages", type=int, default=0, metavar="T",
                    help="only run R/K/P/U at this T a few times (for ncu captures)")
    ap.add_argument("--probe-topk", type=int, default=0, metavar="T",
                    help="only run moe_topk_route at this T a few times (for ncu captures)")
    ap.add_argument("--probe-layer", type=int, default=0, metavar="T",
                    help="only run moe_layer at this T a few times (for ncu captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # asked for N GPUs without a launcher: start one rank per GPU on this
        # node (torch.distributed.run, rendezvous on 127.0.0.1) and pass rank
        # 0's line through
        sys.exit(spawn_ranks(args.gpus))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus and rank == 0:
        log(f"--gpus {args.gpus} but the launcher started {world} ranks: timing {world}")

    if args.launch_check:
        print_launch_check(rank, world)
        return

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return

    if args.probe_topk:
        from mixture_experts_layer_07_gb300 import synth
        torch.cuda.set_device(local_rank)
        print(json.dumps(probe_topk(synth.SPECS[args.workload], args.probe_topk, 3,
                                    f"cuda:{local_rank}")), flush=True)
        return
    if args.probe_stages:
        from mixture_experts_layer_07_gb300 import synth
        torch.cuda.set_device(local_rank)
        print(json.dumps(probe_stages(synth.SPECS[args.workload], args.probe_stages, 3,
                                      f"cuda:{local_rank}")), flush=True)
        return

    if args.probe_layer:
        from mixture_experts_layer_07_gb300 import synth
        torch.cuda.set_device(local_rank)
        print(json.dumps(probe_layer(workload_spec(args), args.probe_layer, 3,
                                     f"cuda:{local_rank}")), flush=True)
        return

    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        res = run_ours(args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(res), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
