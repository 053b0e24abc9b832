"""moe_permute_static -- the permute for callers that cannot allocate device
memory (a fixed pool or arena owns it all, or the calling hook may not call
cudaMalloc), so they have no scratch buffer to hand over.  Its scratch is a
fixed array inside the library.  Checked through the C ABI against the
scratch-taking moe_permute on the same inputs, on two calls in a row (the
second call reuses the array the first one left behind)."""
import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_layer_07_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ops():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mixture_experts_layer_07_gb300 import build
    build.build()
    from mixture_experts_layer_07_gb300 import ops as o
    return o


def permute_both(ops, T, K, E, H, seed):
    ids = torch.from_numpy(synth.random_ids(T, K, E, seed=seed)).cuda()
    x = torch.randn(T, H, device="cuda", generator=torch.Generator("cuda").manual_seed(seed)).to(torch.bfloat16)
    R = T * K
    outs = []
    for static in (False, True):
        off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
        r2f = torch.full((R,), -7, dtype=torch.int32, device="cuda")
        f2r = torch.full((R,), -7, dtype=torch.int32, device="cuda")
        xp = torch.zeros(R, H, dtype=torch.bfloat16, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        if static:
            ops.permute_static(x, ids, E, off, r2f, f2r, xp, st)
        else:
            scratch = torch.empty(ops.permute_scratch_bytes(T, E, K), dtype=torch.uint8, device="cuda")
            ops.permute(x, ids, E, off, r2f, f2r, xp, scratch, st)
        torch.cuda.synchronize()
        outs.append((off.cpu(), r2f.cpu(), f2r.cpu(), xp.view(torch.int16).cpu(), int(st.item())))
    return outs


# (T, K, E, H, seed).  Decode sizes (T*K <= 4096) take the one-CTA permute,
# which keeps its counts in shared memory; larger ones the count / scan /
# scatter kernels, whose chunk counts live in the built-in array.  4080 x 16
# replicas at E = 1024 is the largest size the array holds (255 chunks of 256).
CASES = [(1, 8, 128, 2048, 3), (8, 8, 128, 2048, 4), (2048, 8, 128, 2048, 1),
         (512, 16, 1024, 64, 2), (4080, 16, 1024, 16, 5)]


@pytest.mark.parametrize("T,K,E,H,seed", CASES)
def test_static_scratch_permute_matches_scratch_permute_twice(ops, T, K, E, H, seed):
    # the same problem twice in a row, then another one: each later call runs
    # on what the earlier one left in the built-in array
    if T * K == 65280:
        assert ops.permute_scratch_bytes(T, E, K) <= ops.PERMUTE_STATIC_SCRATCH_BYTES
    for s in (seed, seed, seed + 100):
        a, b = permute_both(ops, T, K, E, H, s)
        assert a[4] == 0 and b[4] == 0
        for u, v in zip(a[:4], b[:4]):
            assert torch.equal(u, v)   # integer and copied bytes: bit for bit


def test_static_scratch_rejects_sizes_beyond_its_maximum(ops):
    T, K, E = 4081, 16, 1024       # one replica past 255 chunks: 256 x 1024 x 4 B > 1 MiB
    assert ops.permute_scratch_bytes(T, K=K, E=E) > ops.PERMUTE_STATIC_SCRATCH_BYTES
    rc = ops.lib().moe_permute_static(None, 0x1000, T, 64, E, K, 0x1000, 0x1000, 0x1000, None,
                                      None, None)
    assert rc == 3  # MOE_ERR_WORKSPACE, before anything is queued
