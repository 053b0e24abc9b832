"""Routing device code run on the CPU, without a GPU.

Each program under tests/host_emu/ includes simt_emu.h (a CTA as host threads:
warp collectives meet at a warp barrier, __syncthreads at a CTA barrier) and
then the device headers themselves, so the CUDA source runs lane by lane on
the host:

* topk_emu.cpp -- csrc/topk_group.cuh and csrc/topk_warp.cuh against a stable
  sort of the same keys (random, tie-heavy, one-lane-owns-every-pick and
  all-tied-in-one-lane logits; float4 and scalar rows; groups of 8, 16 and 32
  lanes and one warp per token; both score modes);
* permute_plan_emu.cpp -- csrc/permute_block.cuh and csrc/plan.cuh (the
  one-CTA permute and GEMM plan of the fused routing launches) against a
  stable counting sort and the work lists the variants imply, with
  out-of-range ids flagged.

This pins the routing logic itself; the GPU parity tests pin the compiled
kernels."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
EMU = os.path.join(ROOT, "tests", "host_emu")


def _cuda_include():
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH") or "/usr/local/cuda"
    inc = os.path.join(home, "include")
    return inc if os.path.exists(os.path.join(inc, "cuda_runtime.h")) else None


@pytest.mark.parametrize("program", ["topk_emu", "permute_plan_emu"])
def test_routing_device_code_on_host(tmp_path, program):
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
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout[-3000:]
