"""The top-K device code (csrc/topk_group.cuh, csrc/topk_warp.cuh) run on the CPU.

tests/host_emu/topk_emu.cpp compiles those headers with the host C++
compiler, runs one warp as 32 threads whose warp intrinsics meet at barriers,
and checks the picks against a stable sort of the same keys (random,
tie-heavy, and one-lane-owns-every-pick logits; float4 and scalar rows; groups
of 8, 16 and 32 lanes and one warp per token; both score modes).  No GPU is
involved: this pins the routing logic itself, while the GPU parity tests pin
the compiled kernels."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_include():
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH") or "/usr/local/cuda"
    inc = os.path.join(home, "include")
    return inc if os.path.exists(os.path.join(inc, "cuda_runtime.h")) else None


def test_topk_logic_on_host(tmp_path):
    cxx = shutil.which("g++")
    inc = _cuda_include()
    if not cxx or not inc:
        pytest.skip("needs g++ and the CUDA headers")
    exe = tmp_path / "topk_emu"
    src = os.path.join(ROOT, "tests", "host_emu", "topk_emu.cpp")
    cmd = [cxx, "-std=c++20", "-O1", "-ffp-contract=off", "-I", inc,
           "-I", os.path.join(ROOT, "mixture_experts_layer_07_gb300", "csrc"),
           "-I", os.path.join(ROOT, "include"), src, "-o", str(exe), "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout[-3000:]
