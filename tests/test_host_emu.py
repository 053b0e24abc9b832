"""Routing device code run on the CPU, without a GPU.

Each program under tests/host_emu/ includes simt_emu.h (a CTA as host threads:
warp collectives meet at a warp barrier, __syncthreads at a CTA barrier) and
then the device headers themselves, so the CUDA source runs lane by lane on
the host:

* topk_emu.cpp -- csrc/topk_group.cuh and csrc/topk_warp.cuh against a stable
  sort of the same keys (random, tie-heavy, one-lane-owns-every-pick and
  all-tied-in-one-lane logits; float4 and scalar rows; groups of 8, 16 and 32
  lanes and one warp per token; both score modes);
* topk_thread_emu.cpp -- csrc/topk_thread.cuh (the thread-per-token route
  of large batches with E <= 128: a bound from group maxima, then only the
  experts above it inserted) against a stable sort of the same keys, for
  every list length, float4 and scalar rows, both score modes and random,
  tie-heavy, all-equal and every-pick-in-one-group logits;
* permute_plan_emu.cpp -- csrc/permute_block.cuh and csrc/plan.cuh (the
  one-CTA permute and GEMM plan of the fused routing launches) against a
  stable counting sort and the work lists the variants imply, with
  out-of-range ids flagged;
* gemv_route_emu.cpp -- csrc/gemv_route.cuh (the matrix-vector decode path's
  routing inside each G1 CTA: a warp per token for E <= 128, slices of the
  experts over 8 / T' warps and a merge beyond; a one-warp stable
  permutation and the skinny plan) against a stable sort, a counting sort,
  the plan's definition and moe_variant_of, as CTA 0 (writing the workspace)
  and as another CTA, both score modes, random and tie-heavy logits.

* sigmoid_emu.cpp -- the selection key's float32 sigmoid (sigmoid_key), the
  order-preserving key map (order_key) and its inverse (key_float) of
  csrc/topk_warp.cuh, compared bit for bit with the oracle's float32 sigmoid,
  with float order and with the inputs.

This pins the routing logic itself; the GPU parity tests pin the compiled
kernels."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
EMU = os.path.join(ROOT, "tests", "host_emu")


def _cuda_include():
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH") or "/usr/local/cuda"
    inc = os.path.join(home, "include")
    return inc if os.path.exists(os.path.join(inc, "cuda_runtime.h")) else None


def _compile(tmp_path, program):
    cxx = shutil.which("g++")
    inc = _cuda_include()
    if not cxx or not inc:
        pytest.skip("needs g++ and the CUDA headers")
    exe = tmp_path / program
    cmd = [cxx, "-std=c++20", "-O1", "-ffp-contract=off", "-I", inc, "-I", EMU,
           "-I", os.path.join(ROOT, "mixture_experts_layer_07_gb300", "csrc"),
           "-I", os.path.join(ROOT, "include"), os.path.join(EMU, program + ".cpp"),
           "-o", str(exe), "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    return str(exe)


@pytest.mark.parametrize("program", ["topk_emu", "topk_thread_emu", "permute_plan_emu",
                                     "gemv_route_emu"])
def test_routing_device_code_on_host(tmp_path, program):
    exe = _compile(tmp_path, program)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout[-3000:]


def test_selection_key_formula_on_host(tmp_path):
    # both sides evaluate one float32 formula op by op, so the device source's
    # bits must equal the oracle's on every input, saturation edges included
    exe = _compile(tmp_path, "sigmoid_emu")
    x = np.linspace(-95, 95, 100001, dtype=np.float32)
    x = np.concatenate([x, np.float32([0.0, -0.0, 1e-30, -1e-30, 87.0, -87.0, 88.0, -88.0,
                                       88.5, -88.5, np.inf, -np.inf])])
    inp = "\n".join(str(int(b)) for b in x.view(np.uint32)) + "\n"
    r = subprocess.run([exe], input=inp, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    out = np.array([[int(v) for v in ln.split()] for ln in r.stdout.split("\n") if ln],
                   dtype=np.uint64)
    sig = out[:, 0].astype(np.uint32)
    ref = oracle.sigmoid_f32(x[np.isfinite(x)]).view(np.uint32)
    assert np.array_equal(sig[np.isfinite(x)], ref)
    # order_key: monotone in float order, -0 and +0 equal, and never 0
    key = out[:, 1].astype(np.uint32)
    order = np.argsort(x, kind="stable")
    xs, ks = x[order], key[order]
    assert (np.diff(ks.astype(np.int64)) >= 0).all()
    assert ((np.diff(ks.astype(np.int64)) == 0) == (np.diff(xs) == 0)).all()
    assert (key != 0).all()
    # key_float inverts order_key exactly (-0 comes back as +0)
    back = out[:, 2].astype(np.uint32).view(np.float32)
    want = np.where(x == 0, np.float32(0.0), x)
    assert np.array_equal(back.view(np.uint32), want.view(np.uint32))
