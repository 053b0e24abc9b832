"""The C-ABI library loads, exports every declared symbol, and rejects bad
arguments on the host (no GPU needed: every call here fails validation
before anything is queued, or is a host-only helper)."""
import ctypes
import json
import os
import re

import pytest

from mixture_experts_layer_07_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")


@pytest.fixture(scope="module")
def ops():
    build_mod.build()
    from mixture_experts_layer_07_gb300 import ops as o
    return o


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_stage_entry_points():
    names = declared_functions()
    for n in ("moe_router_gemm", "moe_topk_route", "moe_permute", "moe_grouped_gemm",
              "moe_unpermute", "moe_layer", "moe_workspace_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(ops):
    lib = ctypes.CDLL(ops.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert set(ops.EXPORTS) <= set(declared_functions())


def test_status_strings(ops):
    assert ops.status_string(0) == "ok"
    assert ops.status_string(3) == "scratch or workspace too small"
    assert ops.status_string(99) == "unknown status"


def test_block_variant_golden_predicate(ops):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "dispatch_predicate.json")))
    thr = g["threshold"]
    # the pages' predicate is two-way (small block / large tile); on the GPU the
    # large side is split again by size (128- or 256-row token tiles)
    large = {ops.VARIANT_TILE, ops.VARIANT_WIDE}

    def pages_code(v):
        return 2 if v in large else v

    for m, want in g["per_block"]:
        assert pages_code(ops.block_variant(m, 1 << 20, 8, thr, ops.DISPATCH_PER_BLOCK)) == want, m
    w = g["worked"]
    off = w["offsets"]
    R, E = off[-1], w["E"]
    sizes = [off[i + 1] - off[i] for i in range(E)]
    assert [pages_code(ops.block_variant(m, R, E, thr, ops.DISPATCH_PER_BLOCK)) for m in sizes] == \
        w["per_block_variants"]
    assert [pages_code(ops.block_variant(m, R, E, thr, ops.DISPATCH_GLOBAL_AVG)) for m in sizes] == \
        w["global_average_variants"]
    assert ops.block_variant(128, R, E, thr, 0, ops.W_FP8) == ops.VARIANT_TILE
    assert ops.block_variant(129, R, E, thr, 0, ops.W_FP8) == ops.VARIANT_WIDE
    assert ops.block_variant(4096, R, E, thr, 0, ops.W_FP8) == ops.VARIANT_WIDE
    assert ops.block_variant(4096, R, E, thr, 0, ops.W_BF16) == ops.VARIANT_TILE
    assert ops.block_variant(3, R, E, thr, ops.DISPATCH_SIMT) == ops.VARIANT_SIMT
    assert ops.block_variant(0, R, E, thr, ops.DISPATCH_SIMT) == ops.VARIANT_SKIP
    assert ops.default_m_skinny() > 0
    assert ops.block_variant(ops.default_m_skinny(), R, E) == ops.VARIANT_SKINNY
    assert ops.block_variant(ops.default_m_skinny() + 1, R, E) == ops.VARIANT_TILE


def _cfg(ops, **kw):
    base = dict(T_max=64, H=256, E=8, K=2, I=128)
    base.update(kw)
    return ops.make_config(**base)


def test_workspace_sizes_grow_with_t_max(ops):
    a = ops.workspace_bytes(_cfg(ops, T_max=16))
    b = ops.workspace_bytes(_cfg(ops, T_max=1024))
    assert 0 < a < b
    L = ops.workspace_layout(_cfg(ops, T_max=16))
    offs = [L.logits, L.ids, L.weights, L.shared_gate, L.offsets, L.row_to_flat, L.flat_to_row,
            L.xp, L.hact, L.y, L.block_variant, L.permute_scratch, L.gemm_scratch]
    assert all(o % 256 == 0 for o in offs)
    assert offs == sorted(offs) and L.total == a
    # the permuted activations hold T_max*K rows of H bf16
    assert L.hact - L.xp >= 16 * 2 * 256 * 2
    assert ops.permute_scratch_bytes(2048, 128, 8) >= 64 * 128 * 4
    assert ops.grouped_gemm_scratch_bytes(16384, 128) > ops.grouped_gemm_scratch_bytes(16, 128)


@pytest.mark.parametrize("kw", [dict(H=100), dict(K=0), dict(K=9), dict(E=2048), dict(I=10),
                                dict(mode=5), dict(wdtype=7), dict(dispatch=9), dict(dispatch=5),
                                dict(m_skinny=-2), dict(has_shared=True, I_shared=0),
                                dict(K=33, E=64)])
def test_config_validation(ops, kw):
    with pytest.raises(ops.MoEError) as ei:
        ops.workspace_bytes(_cfg(ops, **kw))
    assert ei.value.code in (1, 2)


def call(ops, name, *args):
    return getattr(ops.lib(), name)(*args)


def test_router_gemm_rejects_bad_arguments(ops):
    assert call(ops, "moe_router_gemm", 0x1000, 0x1000, None, 0x1000, -1, 64, 8, None) == 1
    assert call(ops, "moe_router_gemm", 0x1000, 0x1000, None, 0x1000, 4, 60, 8, None) == 1
    assert call(ops, "moe_router_gemm", None, 0x1000, None, 0x1000, 4, 64, 8, None) == 1
    assert call(ops, "moe_router_gemm", 0x1008, 0x1000, None, 0x1000, 4, 64, 8, None) == 4
    assert call(ops, "moe_router_gemm", 0x1000, 0x1000, None, 0x1000, 0, 64, 8, None) == 0


def test_router_gemm_tc_rejects_bad_arguments(ops):
    need = ops.router_tc_scratch_bytes(64, 8)
    assert need >= 3 * 64 * 8 * 2
    f = "moe_router_gemm_tc"

    def r(x=0x1000, T=4, H=64, scratch=0x10000, nbytes=need):
        return call(ops, f, x, 0x1000, None, 0x1000, T, H, 8, scratch, nbytes, None, None)

    assert r(H=60) == 1
    assert r(scratch=None) == 1
    assert r(x=None) == 1
    assert r(nbytes=need - 1) == 3
    assert r(scratch=0x10010) == 4
    assert r(x=0x1008) == 4
    assert r(T=0) == 0
    with pytest.raises(ops.MoEError):
        ops.router_tc_scratch_bytes(60, 8)


def test_topk_route_rejects_bad_arguments(ops):
    f = "moe_topk_route"
    assert call(ops, f, 0x1000, 8, None, 4, 8, 9, 0, 1.0, 0x1000, 0x1000, None, None) == 1
    assert call(ops, f, 0x1000, 7, None, 4, 8, 2, 0, 1.0, 0x1000, 0x1000, None, None) == 1
    assert call(ops, f, 0x1000, 8, None, 4, 8, 2, 0, 1.0, 0x1000, 0x1000, 0x1000, None) == 1
    assert call(ops, f, 0x1000, 8, None, 4, 8, 2, 3, 1.0, 0x1000, 0x1000, None, None) == 1
    assert call(ops, f, 0x1001, 8, None, 4, 8, 2, 0, 1.0, 0x1000, 0x1000, None, None) == 4
    assert call(ops, f, 0x1000, 8, None, 0, 8, 2, 0, 1.0, 0x1000, 0x1000, None, None) == 0


def test_permute_rejects_short_or_misaligned_scratch(ops):
    need = ops.permute_scratch_bytes(64, 8, 2)
    f = "moe_permute"
    args = [0x1000, 0x1000, 64, 256, 8, 2, 0x1000, 0x1000, 0x1000, 0x1000]
    assert call(ops, f, *args, 0x10000, need - 1, None, None) == 3
    assert call(ops, f, *args, 0x10010, need, None, None) == 4
    assert call(ops, f, *args, None, need, None, None) == 1
    bad = list(args)
    bad[5] = 9  # K > E
    assert call(ops, f, *bad, 0x10000, need, None, None) == 1


def test_grouped_gemm_rejects_bad_arguments(ops):
    need = ops.grouped_gemm_scratch_bytes(32, 8)
    f = "moe_grouped_gemm"

    def g(R=32, H=256, I=128, wdtype=0, w=0x1000, s=None, scratch=0x10000, nbytes=need,
          m_skinny=-1, dispatch=0):
        return call(ops, f, 0x1000, 0x1000, 8, R, H, I, wdtype, w, w, w, s, s, s, 0x1000, 0x1000,
                    m_skinny, dispatch, None, scratch, nbytes, None, None)

    assert g(H=200) == 1
    assert g(I=72) == 1
    assert g(wdtype=4) == 2
    assert g(wdtype=1) == 1          # FP8 without scales
    assert g(wdtype=2) == 1          # MXFP4 without scales
    assert g(wdtype=2, H=240, s=0x1000) == 1  # MXFP4 rows hold whole 32-element blocks
    assert g(wdtype=2, I=144, s=0x1000) == 1
    assert g(nbytes=need - 16) == 3
    assert g(scratch=0x10040) == 4
    assert g(w=0x1002) == 4
    assert g(m_skinny=-3) == 1
    assert g(dispatch=3) == 1
    assert g(dispatch=4) == 1          # the GEMV decode path is a moe_layer option


def test_unpermute_rejects_bad_arguments(ops):
    f = "moe_unpermute"
    assert call(ops, f, 0x1000, 0x1000, 0x1000, 4, 2, 250, None, None, 0x1000, None) == 1
    assert call(ops, f, 0x1000, 0x1000, 0x1000, 4, 2, 256, 0x1000, None, 0x1000, None) == 1
    assert call(ops, f, 0x1004, 0x1000, 0x1000, 4, 2, 256, None, None, 0x1000, None) == 4
    assert call(ops, f, 0x1000, 0x1000, 0x1000, 0, 2, 256, None, None, 0x1000, None) == 0


def test_layer_rejects_bad_arguments(ops):
    cfg = _cfg(ops)
    need = ops.workspace_bytes(cfg)
    w = ops.Weights(0x1000, None, None, 0x1000, 0x1000, 0x1000, None, None, None, None, None, None)
    lib = ops.lib()
    by = ctypes.byref
    assert lib.moe_layer(by(cfg), 65, 0x1000, by(w), 0x1000, 0x10000, need, None, None) == 1
    assert lib.moe_layer(by(cfg), 8, 0x1000, by(w), 0x1000, 0x10000, need - 1, None, None) == 3
    assert lib.moe_layer(by(cfg), 8, 0x1000, by(w), 0x1000, 0x10080, need, None, None) == 4
    assert lib.moe_layer(by(cfg), 0, 0x1000, by(w), 0x1000, 0x10000, need, None, None) == 0
    fp8 = _cfg(ops, wdtype=1)
    assert lib.moe_layer(by(fp8), 8, 0x1000, by(w), 0x1000, 0x10000,
                         ops.workspace_bytes(fp8), None, None) == 1
    mx = _cfg(ops, wdtype=2)
    assert lib.moe_layer(by(mx), 8, 0x1000, by(w), 0x1000, 0x10000,
                         ops.workspace_bytes(mx), None, None) == 1
    sh = _cfg(ops, has_shared=True, I_shared=64)
    assert lib.moe_layer(by(sh), 8, 0x1000, by(w), 0x1000, 0x10000,
                         ops.workspace_bytes(sh), None, None) == 1


def test_bounded_wait_check_rejects_bad_arguments(ops):
    f = "moe_bounded_wait_check"
    assert call(ops, f, None, 1, 1000, 0x1000, None) == 1
    assert call(ops, f, 0x1000, 1, 1000, None, None) == 1
    assert call(ops, f, 0x1000, 1, 0, 0x1000, None) == 1
    assert call(ops, f, 0x1000, 1, 10000001, 0x1000, None) == 1


def test_one_launch_dispatch_is_a_layer_option(ops):
    # MOE_DISPATCH_ONE_LAUNCH is accepted by the layer's config (same
    # workspace as per-block dispatch) and refused by the stand-alone grouped
    # GEMM (checked in test_grouped_gemm_rejects_bad_arguments)
    a = ops.workspace_bytes(_cfg(ops, dispatch=ops.DISPATCH_ONE_LAUNCH))
    b = ops.workspace_bytes(_cfg(ops))
    assert a == b > 0
    # so is MOE_DISPATCH_GEMV, except with W8A8 (tensor cores only)
    assert ops.workspace_bytes(_cfg(ops, dispatch=ops.DISPATCH_GEMV)) == b
    with pytest.raises(ops.MoEError):
        ops.workspace_bytes(_cfg(ops, dispatch=ops.DISPATCH_GEMV, wdtype=ops.W8A8_FP8))
