"""GPU parity: every stage of the CUDA path through the C ABI, element by
element against the CPU oracle on the same seeded inputs (tolerances in
tests/gpu_util.py).  Sizes span several tiles and a ragged tail; full-size
workloads are checked on sampled tokens in test_gpu_fullsize.py."""
import time

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_07_gb300 import synth
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

SPECS = synth.SPECS


@pytest.fixture(scope="module")
def ops():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from mixture_experts_layer_07_gb300 import build
    build.build()
    from mixture_experts_layer_07_gb300 import ops as o
    return o


def sync():
    torch.cuda.synchronize()


def i32(n):
    return torch.empty(n, dtype=torch.int32, device="cuda")


# ---------------------------------------------------------------- R
ROUTER_CASES = [("tiny", 16), ("qwen3_30b_a3b", 1), ("qwen3_30b_a3b", 8),
                ("qwen3_30b_a3b", 17), ("qwen3_30b_a3b", 256), ("gpt_oss_20b", 32),
                ("shared_gate", 4), ("shared_gate", 131), ("high_expert", 512)]


@pytest.mark.parametrize("name,T", ROUTER_CASES)
def test_router_gemm(ops, name, T):
    spec = SPECS[name]
    inp = synth.host_inputs(spec, T, seed=1, weights=False)
    logits = torch.full((T, spec.G), float("nan"), device="cuda")
    ops.router_gemm(U.bf16_dev(inp["x_bits"]), U.dev(inp["wg"]), U.dev(inp["gate_bias"]), logits)
    sync()
    U.assert_router_close(U.f64(logits), oracle.bf16_to_f64(inp["x_bits"]), inp["wg"],
                          inp["gate_bias"])


# tensor-core router: the same bound, from the bf16 three-way weight split;
# cases cover one and two 128-token halves per CTA, split-K clusters, several
# gate tiles, G = E + 1, a K tail below the 64-wide step and T below one tile
ROUTER_TC_CASES = [("tiny", 1), ("tiny", 16), ("qwen3_30b_a3b", 64), ("qwen3_30b_a3b", 2125),
                   ("qwen3_30b_a3b", 9733), ("gpt_oss_20b", 300), ("shared_gate", 131),
                   ("high_expert", 4100), ("ragged_h", 200)]


def router_tc_spec(name):
    if name == "ragged_h":
        return SPECS["tiny"].with_(name="ragged_h", H=136, E=40, K=4)
    return SPECS[name]


@pytest.mark.parametrize("name,T", ROUTER_TC_CASES)
def test_router_gemm_tc(ops, name, T):
    spec = router_tc_spec(name)
    inp = synth.host_inputs(spec, T, seed=3, weights=False)
    x, wg, gb = U.bf16_dev(inp["x_bits"]), U.dev(inp["wg"]), U.dev(inp["gate_bias"])
    scratch = torch.empty(ops.router_tc_scratch_bytes(spec.H, spec.G), dtype=torch.uint8,
                          device="cuda")
    st = i32(1).zero_()
    logits = torch.full((T, spec.G), float("nan"), device="cuda")
    ops.router_gemm_tc(x, wg, gb, logits, scratch, st)
    sync()
    assert st.item() == 0
    U.assert_router_close(U.f64(logits), oracle.bf16_to_f64(inp["x_bits"]), inp["wg"],
                          inp["gate_bias"])
    # deterministic: the same bits on a second call
    again = torch.full_like(logits, float("nan"))
    ops.router_gemm_tc(x, wg, gb, again, scratch, st)
    sync()
    assert torch.equal(logits, again)


def test_router_gemm_tc_extreme_weights(ops):
    # weights spanning many binades (the split must carry each one's own 24
    # bits) and exact zeros
    spec = SPECS["tiny"]
    T = 130
    inp = synth.host_inputs(spec, T, seed=5, weights=False)
    rng = np.random.default_rng(11)
    wg = (inp["wg"].astype(np.float64) * 2.0 ** rng.integers(-40, 40, inp["wg"].shape))
    wg[:, ::7] = 0.0
    wg = wg.astype(np.float32)
    logits = torch.empty((T, spec.G), device="cuda")
    scratch = torch.empty(ops.router_tc_scratch_bytes(spec.H, spec.G), dtype=torch.uint8,
                          device="cuda")
    ops.router_gemm_tc(U.bf16_dev(inp["x_bits"]), U.dev(wg), None, logits, scratch)
    sync()
    U.assert_router_close(U.f64(logits), oracle.bf16_to_f64(inp["x_bits"]), wg)


# ---------------------------------------------------------------- K
TOPK_CASES = [  # E, K, mode, T, shared
    (8, 2, 0, 16, False), (128, 8, 0, 1, False), (128, 8, 0, 2048, False),
    (32, 4, 0, 517, False), (512, 10, 0, 64, True), (896, 16, 1, 512, False),
    (512, 9, 1, 512, False), (1024, 16, 1, 512, False), (1024, 9, 1, 37, False),
    (512, 16, 1, 512, False), (1024, 9, 1, 512, False), (512, 16, 0, 512, True),
    (8, 8, 0, 5, False), (64, 32, 0, 3, False), (33, 3, 1, 70, True), (1, 1, 0, 4, False),
    # large T: many CTAs of four token warps
    (128, 8, 0, 5000, False), (32, 4, 0, 4096, False), (256, 16, 1, 4100, True),
    (8, 2, 0, 4097, False), (200, 9, 1, 8191, False),
    # E <= 128 at T >= 32768: groups of 8 lanes per token (float4 rows and,
    # with a shared-gate column, scalar rows)
    (128, 8, 0, 40000, False), (32, 4, 0, 33000, False), (64, 6, 1, 33000, True),
    (100, 7, 0, 32768, False), (33, 3, 1, 40000, True), (64, 32, 0, 32768, False),
    (8, 8, 1, 32770, False)]


def run_topk(ops, logits, E, K, mode, scale, sel_bias, shared):
    T = logits.shape[0]
    ids = i32((T, K))
    w = torch.empty(T, K, device="cuda")
    gsh = torch.empty(T, device="cuda") if shared else None
    ops.topk_route(U.dev(logits), E, K, mode, scale, ids, w, U.dev(sel_bias), gsh)
    sync()
    return ids.cpu().numpy(), w.cpu().numpy(), None if gsh is None else gsh.cpu().numpy()


@pytest.mark.parametrize("E,K,mode,T,shared", TOPK_CASES)
def test_topk_route(ops, E, K, mode, T, shared):
    G = E + int(shared)
    lg = synth.random_logits(T, G, seed=E * 31 + K)
    scale = 2.5 if mode else 1.0
    bias = synth._normal(7, 9, E, (E,), 0.1 ** 0.5) if mode else None
    ids, w, gsh = run_topk(ops, lg, E, K, mode, scale, bias, shared)
    if mode == 0:
        rid, rw = oracle.topk_softmax_renorm(lg.astype(np.float64), E, K)
    else:
        rid, rw = oracle.topk_sigmoid_bias(lg, bias, E, K, scale)
    assert np.array_equal(ids, rid)
    U.assert_weights_close(w, rw)
    if shared:
        U.assert_weights_close(gsh, oracle.shared_gate(lg.astype(np.float64), E))


@pytest.mark.parametrize("mode,T", [(0, 300), (1, 300), (0, 5000), (1, 5000), (0, 40000),
                                    (1, 40000)])
def test_topk_heavy_ties(ops, mode, T):
    # logits from a 3-value set: most keys tie, the index rule decides
    E, K = 128, 8
    r = np.random.default_rng(3)
    lg = r.choice(np.float32([-1.0, 0.0, 1.0]), size=(T, E)).astype(np.float32)
    lg[0] = 0.5                                   # one all-equal row
    lg[1] = -0.0
    lg[1, ::2] = 0.0                              # -0 and +0 are equal keys
    bias = np.zeros(E, np.float32) if mode else None
    ids, w, _ = run_topk(ops, lg, E, K, mode, 2.5 if mode else 1.0, bias, False)
    if mode == 0:
        rid, rw = oracle.topk_softmax_renorm(lg.astype(np.float64), E, K)
    else:
        rid, rw = oracle.topk_sigmoid_bias(lg, bias, E, K, 2.5)
    assert np.array_equal(ids, rid)
    assert ids[0].tolist() == list(range(K)) and ids[1].tolist() == list(range(K))
    U.assert_weights_close(w, rw)


@pytest.mark.parametrize("E,K,G,T", [(128, 8, 128, 40000), (128, 8, 129, 40000),
                                     (896, 16, 896, 600), (1024, 16, 1024, 300),
                                     (256, 16, 257, 700)])
def test_topk_top_experts_on_one_lane(ops, E, K, G, T):
    # every token's top 2K logits sit on the experts one lane of a routing
    # group owns, under both lane layouts (float4 rows: lane q of a group of
    # GS owns e with (e % 4GS) // 4 == q; scalar rows: e % GS == q), so that
    # lane supplies all K picks and must rebuild its candidate list
    GS = 8 if E <= 128 else 16 if E <= 256 else 32
    r = np.random.default_rng(E + G)
    lg = r.standard_normal((T, G)).astype(np.float32)
    e = np.arange(E)
    for t in range(T):
        q = t % GS
        own = (e % (4 * GS)) // 4 == q if G % 4 == 0 else e % GS == q
        sel = e[own][:2 * K]
        lg[t, sel] = 10.0 + r.standard_normal(len(sel)).astype(np.float32)
    ids, w, _ = run_topk(ops, lg, E, K, 0, 1.0, None, False)
    rid, rw = oracle.topk_softmax_renorm(lg.astype(np.float64), E, K)
    assert np.array_equal(ids, rid)
    U.assert_weights_close(w, rw)


def test_sigmoid_key_selection_order_matches_oracle(ops):
    # the selection key is one specified float32 formula on both sides; a
    # K = E route over a dense sweep of logits makes the GPU's selection order
    # the order of its keys, which must equal the oracle's order of its keys
    # (the keys' bits themselves are compared on the host, where the device
    # header is compiled and run against the oracle: tests/test_host_emu.py)
    E = 32
    lg = np.linspace(-95, 95, 32 * 4001, dtype=np.float32).reshape(-1, E)
    ids, _, _ = run_topk(ops, lg, E, E, 1, 1.0, np.zeros(E, np.float32), False)
    rid, _ = oracle.topk_sigmoid_bias(lg, np.zeros(E, np.float32), E, E, 1.0)
    assert np.array_equal(ids, rid)
    # sigmoid_f32 agrees with CUDA's expf-based sigmoid to a few ulp
    t = torch.from_numpy(lg).cuda()
    ref = (1.0 / (1.0 + torch.exp(-t))).cpu().numpy()
    mine = oracle.sigmoid_f32(lg)
    ok = ref > 1e-30
    assert (np.abs(mine[ok] - ref[ok]) <= 4 * np.spacing(ref[ok])).all()


# ---------------------------------------------------------------- P
PERMUTE_CASES = [(16, 2, 8, 256), (1, 8, 128, 2048), (37, 8, 128, 2048), (2048, 8, 128, 2048),
                 (4096, 4, 32, 2880), (512, 16, 896, 64), (512, 16, 1024, 64), (64, 10, 512, 2048),
                 (33, 1, 3, 16), (20000, 4, 32, 64), (9000, 8, 128, 16), (5000, 16, 1024, 16)]


def run_permute(ops, x, ids, E, want_xp=True):
    T, K = ids.shape
    R = T * K
    H = x.shape[1]
    off, r2f, f2r = i32(E + 1), i32(R), i32(R)
    xp = torch.empty(R, H, dtype=torch.bfloat16, device="cuda") if want_xp else None
    scratch = torch.empty(ops.permute_scratch_bytes(T, E, K), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.permute(x, ids, E, off, r2f, f2r, xp, scratch, st)
    sync()
    return off, r2f, f2r, xp, int(st.item())


@pytest.mark.parametrize("T,K,E,H", PERMUTE_CASES)
def test_permute(ops, T, K, E, H):
    ids = synth.random_ids(T, K, E, seed=T + E)
    x_bits = synth.f32_to_bf16_bits(synth._normal(0, 1, T, (T, H), 1.0))
    x = U.bf16_dev(x_bits)
    off, r2f, f2r, xp, st = run_permute(ops, x, torch.from_numpy(ids).cuda(), E)
    ro, rr, rf = oracle.permute(ids, E)
    assert st == 0
    assert np.array_equal(off.cpu().numpy(), ro)
    assert np.array_equal(r2f.cpu().numpy(), rr)
    assert np.array_equal(f2r.cpu().numpy(), rf)
    got = xp.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, x_bits[rr // K])


def test_permute_concentrated_with_empty_experts(ops):
    T, K, E, H = 300, 4, 32, 64
    r = np.random.default_rng(5)
    ids = np.stack([r.choice([0, 1, 2, 3, 9], size=K, replace=False) for _ in range(T)]).astype(np.int32)
    x = torch.randn(T, H, device="cuda").to(torch.bfloat16)
    off, r2f, f2r, _, st = run_permute(ops, x, torch.from_numpy(ids).cuda(), E)
    ro, rr, rf = oracle.permute(ids, E)
    assert st == 0 and np.array_equal(off.cpu().numpy(), ro)
    assert np.array_equal(r2f.cpu().numpy(), rr) and np.array_equal(f2r.cpu().numpy(), rf)


def test_permute_flags_out_of_range_ids(ops):
    T, K, E = 50, 2, 16
    ids = synth.random_ids(T, K, E, seed=1)
    ids[7, 1] = E        # out of range
    ids[20, 0] = -3
    x = torch.randn(T, 32, device="cuda").to(torch.bfloat16)
    off, r2f, f2r, _, st = run_permute(ops, x, torch.from_numpy(ids).cuda(), E)
    assert st == ops.DEV_BAD_EXPERT_ID
    f2r = f2r.cpu().numpy()
    assert f2r[7 * K + 1] == -1 and f2r[20 * K] == -1
    assert off.cpu().numpy()[-1] == T * K - 2
    valid = np.ones(T * K, bool)
    valid[[7 * K + 1, 20 * K]] = False
    ro, rr, _ = oracle.permute(np.where(valid, ids.ravel(), E), E + 1)
    assert np.array_equal(off.cpu().numpy(), ro[:E + 1])
    assert np.array_equal(r2f.cpu().numpy()[:T * K - 2], rr[:T * K - 2])


def test_permute_then_unpermute_is_identity(ops):
    T, H, E = 129, 256, 8
    x_bits = synth.f32_to_bf16_bits(synth._normal(0, 1, 5, (T, H), 1.0))
    x = U.bf16_dev(x_bits)
    # K = 1 and weight 1: bit-exact round trip
    ids = torch.from_numpy(synth.random_ids(T, 1, E, seed=2)).cuda()
    _, _, f2r, xp, _ = run_permute(ops, x, ids, E)
    out = torch.empty_like(x)
    ops.unpermute(xp, f2r, torch.ones(T, 1, device="cuda"), T, 1, H, out)
    sync()
    assert torch.equal(out.view(torch.int16), x.view(torch.int16))
    # K = 4 with weights summing to 1: within one bf16 rounding
    ids = torch.from_numpy(synth.random_ids(T, 4, E, seed=3)).cuda()
    _, _, f2r, xp, _ = run_permute(ops, x, ids, E)
    w = torch.rand(T, 4, device="cuda")
    w = w / w.sum(1, keepdim=True)
    ops.unpermute(xp, f2r, w, T, 4, H, out)
    sync()
    ref = oracle.bf16_to_f64(x_bits)
    assert (np.abs(U.f64(out) - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30).all()


# ---------------------------------------------------------------- G
def case_id(v):
    """Readable test ids: a spec's overrides as k=v pairs."""
    if isinstance(v, dict):
        return ",".join(f"{k}={x}" for k, x in v.items()) or "base"
    return None


def concentrated_ids(T, K, E, seed):
    """Most tokens pick from a few hot experts (big blocks); the rest spread
    over all experts (small blocks); unpicked experts stay empty."""
    r = np.random.default_rng(seed)
    hot = np.arange(min(E, K + 2))
    rows = [r.choice(hot, K, replace=False) if r.random() < 0.7 else r.choice(E, K, replace=False)
            for _ in range(T)]
    return np.stack(rows).astype(np.int32)


def gemm_case(spec, T, seed, concentrated=False):
    """Host inputs + oracle permute for a grouped-GEMM case."""
    K, E = spec.K, spec.E
    ids = concentrated_ids(T, K, E, seed) if concentrated else synth.random_ids(T, K, E, seed=seed)
    inp = synth.host_inputs(spec, T, seed=seed, experts=sorted(set(ids.ravel().tolist())))
    off, r2f, f2r = oracle.permute(ids, E)
    return inp, ids, off, r2f, f2r


def run_gemm(ops, spec, inp, off, r2f, K, dispatch=0, m_skinny=-1):
    T = inp["x_bits"].shape[0]
    R = T * K
    E, H, I = spec.E, spec.H, spec.I
    xp_bits = inp["x_bits"][r2f // K]
    t = U.layer_tensors(inp, inp["experts"])
    hact = torch.full((R, I), float("nan"), device="cuda").to(torch.bfloat16)
    y = torch.full((R, H), float("nan"), device="cuda").to(torch.bfloat16)
    scratch = torch.empty(ops.grouped_gemm_scratch_bytes(R, E), dtype=torch.uint8, device="cuda")
    bv = i32(E)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.grouped_gemm(U.bf16_dev(xp_bits), torch.from_numpy(off).cuda(), E, H, I, t["w1"], t["w3"],
                     t["w2"], hact, y, scratch, wdtype=U.wdtype_of(ops, spec),
                     s1=t.get("s1"), s3=t.get("s3"), s2=t.get("s2"), m_skinny=m_skinny,
                     dispatch=dispatch, block_variant=bv, dev_status=st)
    sync()
    return hact, y, bv.cpu().numpy(), int(st.item()), xp_bits


GEMM_CASES = [  # spec name, overrides, T, concentrated, dispatch, m_skinny, both variants
    ("tiny", {}, 16, False, 0, -1, False),
    ("tiny", {}, 16, False, 2, -1, False),
    ("qwen3_30b_a3b", {}, 8, False, 0, -1, False),
    ("qwen3_30b_a3b", {}, 256, False, 0, -1, True),
    ("qwen3_30b_a3b", {}, 300, True, 0, -1, True),
    ("qwen3_30b_a3b", {}, 300, True, 1, -1, False),
    ("qwen3_30b_a3b", {}, 300, True, 2, -1, False),
    ("qwen3_30b_a3b", {}, 300, True, 0, 4, True),
    ("tiny", {"H": 2880, "I": 2880, "E": 4}, 40, False, 0, 8, False),
    ("tiny", {"H": 2880, "I": 2880, "E": 4}, 40, False, 0, 64, False),
    ("tiny", {"H": 320, "I": 192, "E": 6}, 200, True, 0, -1, False),
    ("tiny", {"H": 160, "I": 144, "E": 5, "wdtype": "fp8"}, 50, True, 0, -1, False),
    ("tiny", {"H": 160, "I": 144, "E": 5, "wdtype": "fp8"}, 50, True, 2, -1, False),
    # MXFP4 weights (e2m1 pairs + a UE8M0 scale per 32 along each row)
    ("tiny", {"H": 160, "I": 96, "E": 5, "wdtype": "mxfp4"}, 50, True, 0, -1, False),
    ("tiny", {"H": 160, "I": 96, "E": 5, "wdtype": "mxfp4"}, 50, True, 2, -1, False),
    ("gpt_oss_20b", {"wdtype": "mxfp4"}, 40, True, 0, -1, True),
    ("gpt_oss_20b", {"E": 4, "wdtype": "mxfp4"}, 300, True, 0, -1, False),
    ("gpt_oss_20b", {"E": 6, "wdtype": "mxfp4"}, 700, True, 0, -1, False),
    ("tiny", {"H": 2880, "I": 2880, "E": 4, "wdtype": "mxfp4"}, 40, False, 0, 8, False),
    ("gpt_oss_20b", {}, 40, True, 0, -1, True),
    ("gpt_oss_20b", {"E": 6}, 40, True, 2, -1, False),
    ("gpt_oss_20b", {"E": 4}, 300, True, 0, -1, False),
    # blocks of >= 256 rows: the wide (256-row token tile) variant
    ("qwen3_30b_a3b", {}, 1200, True, 0, -1, True),
    ("tiny", {"H": 2880, "I": 2880, "E": 4}, 700, True, 0, -1, False),
    ("gpt_oss_20b", {"E": 6}, 700, True, 0, -1, False),
]


@pytest.mark.parametrize("name,over,T,conc,dispatch,m_skinny,both", GEMM_CASES, ids=case_id)
def test_grouped_gemm(ops, name, over, T, conc, dispatch, m_skinny, both):
    spec = SPECS[name].with_(**over)
    inp, ids, off, r2f, f2r = gemm_case(spec, T, seed=T + spec.E, concentrated=conc)
    hact, y, bv, st, xp_bits = run_gemm(ops, spec, inp, off, r2f, spec.K, dispatch, m_skinny)
    assert st == 0
    w1, w3, w2 = oracle.layer_weights_f64(inp)
    rh, ry = oracle.grouped_gemm(oracle.bf16_to_f64(xp_bits), off, w1, w3, w2)
    rel = 5e-2 if spec.wdtype == "fp8" else 2e-2
    U.assert_bf16_close(U.f64(hact), rh, rel, "hact")
    U.assert_bf16_close(U.f64(y), ry, rel, "y")
    R = T * spec.K
    m = np.diff(off)
    wd = U.wdtype_of(ops, spec)
    want_bv = [ops.block_variant(int(mm), R, spec.E, m_skinny, dispatch, wd) for mm in m]
    assert bv.tolist() == want_bv
    if both:  # small and large blocks in the same call
        assert ops.VARIANT_SKINNY in bv.tolist()
        assert {ops.VARIANT_TILE, ops.VARIANT_WIDE} & set(bv.tolist())
    if dispatch == 0 and spec.wdtype != "bf16" and (m >= ops.WIDE_MIN_ROWS).any():
        assert ops.VARIANT_WIDE in bv.tolist()


def _mx_pack(codes):
    """[rows, cols] e2m1 codes -> [rows, cols / 2] bytes, element 2i low nibble."""
    c = np.asarray(codes, np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def _mx_test_matrix(rows, cols, s_max, seed):
    """Every e2m1 code in every scale block; scale bytes 0..s_max with the
    corners (0, 1, 126..130, s_max) present."""
    r = np.random.default_rng(seed)
    codes = r.integers(0, 16, size=(rows, cols)).astype(np.uint8)
    codes[:, :16] = np.arange(16, dtype=np.uint8)  # each row: all 16 codes
    sc = r.integers(0, s_max + 1, size=(rows, cols // 32)).astype(np.uint8)
    corners = np.array([0, 1, 126, 127, 128, 129, 130, s_max], np.uint8)
    sc.flat[:len(corners)] = corners
    return _mx_pack(codes), sc


def _mx_const(rows, cols, code, s):
    return (_mx_pack(np.full((rows, cols), code, np.uint8)),
            np.full((rows, cols // 32), s, np.uint8))


@pytest.mark.parametrize("T,m_skinny,dispatch", [(256, -1, 0), (128, -1, 0), (256, 1024, 0),
                                                 (256, -1, 2)])
def test_grouped_gemm_mxfp4_reads_every_code_exactly(ops, T, m_skinny, dispatch):
    # one expert, token t = the one-hot row e_t, so G1 reads single weights:
    # hact[t, i] = silu(w1[i, t]) * w3[i, t] and y[t, h] = sum_i hact[t, i] w2[h, i].
    # (a) w1 = 24 (code 6.0 at scale byte 129: the two-step multiply) and w3 the
    #     codes under test: hact = 24 * w3 exactly (silu(24) is 24 in fp32)
    # (b) w3 = identity: hact = 24 * one-hot, so y = 24 * w2 exactly
    # (c) w3 = 1: hact = bf16(silu(w1)) for the codes under test in w1
    H = I = 256
    x = np.zeros((T, H), np.float32)
    x[np.arange(T), np.arange(T)] = 1.0
    xp = U.bf16_dev(synth.f32_to_bf16_bits(x))
    off = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    scratch = torch.empty(ops.grouped_gemm_scratch_bytes(T, 1), dtype=torch.uint8, device="cuda")

    def run(w1, w3, w2):
        t = {}
        for k, (q, sc) in (("1", w1), ("3", w3), ("2", w2)):
            t["w" + k] = U.dev(q[None])
            t["s" + k] = U.dev(sc[None])
        hact = torch.full((T, I), float("nan"), device="cuda").to(torch.bfloat16)
        y = torch.full((T, H), float("nan"), device="cuda").to(torch.bfloat16)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        ops.grouped_gemm(xp, off, 1, H, I, t["w1"], t["w3"], t["w2"], hact, y, scratch,
                         wdtype=ops.W_MXFP4, s1=t["s1"], s3=t["s3"], s2=t["s2"],
                         m_skinny=m_skinny, dispatch=dispatch, dev_status=st)
        sync()
        assert int(st.item()) == 0
        return U.f64(hact), U.f64(y)

    w24 = _mx_const(I, H, 7, 129)
    assert oracle.dequant_mxfp4(*w24)[0, 0] == 24.0
    # (a)
    q3, s3 = _mx_test_matrix(I, H, 240, seed=T + 1)
    w3 = oracle.dequant_mxfp4(q3, s3)
    hact, _ = run(w24, (q3, s3), _mx_const(H, I, 2, 127))
    assert np.array_equal(hact, 24.0 * w3[:, :T].T)
    # (b)
    eye = np.where(np.eye(I, H, dtype=bool), 2, 0).astype(np.uint8)
    q2, s2 = _mx_test_matrix(H, I, 240, seed=T + 2)
    w2 = oracle.dequant_mxfp4(q2, s2)
    hact, y = run(w24, (_mx_pack(eye), np.full((I, H // 32), 127, np.uint8)), (q2, s2))
    assert np.array_equal(hact, 24.0 * np.eye(T, I))
    assert np.array_equal(y, 24.0 * w2[:, :T].T)
    # (c)
    q1, s1 = _mx_test_matrix(I, H, 130, seed=T + 3)
    w1 = oracle.dequant_mxfp4(q1, s1)[:, :T].T
    hact, _ = run((q1, s1), _mx_const(I, H, 2, 127), _mx_const(H, I, 2, 127))
    ref = w1 / (1.0 + np.exp(-w1))
    assert (np.abs(hact - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-37).all()


W8A8_CASES = [  # spec name, overrides, T, concentrated
    ("tiny", {"H": 160, "I": 144, "E": 5, "wdtype": "fp8", "act": "fp8"}, 50, True),
    ("tiny", {"H": 256, "I": 384, "E": 3, "wdtype": "fp8", "act": "fp8"}, 7, False),
    ("gpt_oss_20b", {"E": 4, "act": "fp8"}, 300, True),
    ("gpt_oss_20b", {"E": 6, "act": "fp8"}, 700, True),
    ("qwen3_30b_a3b", {"wdtype": "fp8", "act": "fp8"}, 256, False),
]


@pytest.mark.parametrize("name,over,T,conc", W8A8_CASES, ids=case_id)
def test_grouped_gemm_w8a8(ops, name, over, T, conc):
    # W8A8: the quantised activations the kernels wrote (read back from the
    # scratch) equal the oracle's quantisation of the same bf16 rows bit for
    # bit -- xp before G1, the GPU's own hact before G2; each GEMM matches the
    # oracle applied to the GPU's own quantised input; and the whole call
    # matches the oracle's W8A8 grouped GEMM end to end
    spec = SPECS[name].with_(**over)
    E, H, I, K = spec.E, spec.H, spec.I, spec.K
    inp, ids, off, r2f, f2r = gemm_case(spec, T, seed=T + E + 1, concentrated=conc)
    R = T * K
    xp_bits = inp["x_bits"][r2f // K]
    t = U.layer_tensors(inp, inp["experts"])
    wd = ops.W8A8_FP8
    hact = torch.full((R, I), float("nan"), device="cuda").to(torch.bfloat16)
    y = torch.full((R, H), float("nan"), device="cuda").to(torch.bfloat16)
    plan = ops.grouped_gemm_scratch_bytes(R, E)
    scratch = torch.zeros(ops.grouped_gemm_scratch_bytes(R, E, H, I, wd), dtype=torch.uint8,
                          device="cuda")
    bv = i32(E)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops.grouped_gemm(U.bf16_dev(xp_bits), torch.from_numpy(off).cuda(), E, H, I, t["w1"],
                     t["w3"], t["w2"], hact, y, scratch, wdtype=wd, s1=t["s1"], s3=t["s3"],
                     s2=t["s2"], block_variant=bv, dev_status=st)
    sync()
    assert int(st.item()) == 0
    assert bv.cpu().numpy().tolist() == [ops.VARIANT_TILE if m else ops.VARIANT_SKIP
                                         for m in np.diff(off)]
    # the scratch after the plan: xq [R,H], sx [R,KB1], hq [R,I], sh [R,KB2]
    a256 = lambda n: -(-n // 256) * 256  # noqa: E731
    kb1, kb2 = -(-H // 128), -(-I // 128)
    sc = scratch.cpu().numpy()[plan:]
    o = 0
    xq = sc[o:o + R * H].reshape(R, H); o += a256(R * H)
    sx = sc[o:o + R * kb1 * 4].view(np.float32).reshape(R, kb1); o += a256(R * kb1 * 4)
    hq = sc[o:o + R * I].reshape(R, I); o += a256(R * I)
    sh = sc[o:o + R * kb2 * 4].view(np.float32).reshape(R, kb2)
    x64 = oracle.bf16_to_f64(xp_bits)
    rq, rs = oracle.quantize_act_fp8(x64)
    assert np.array_equal(sx, rs) and np.array_equal(xq, rq)
    h_gpu = U.f64(hact)
    hq_ref, sh_ref = oracle.quantize_act_fp8(h_gpu)
    assert np.array_equal(sh, sh_ref) and np.array_equal(hq, hq_ref)
    # each GEMM on the GPU's own quantised input: fp32 sums and one bf16 rounding
    w1, w3, w2 = oracle.layer_weights_f64(inp)
    xd = oracle.dequant_act_fp8(xq, sx)
    hd = oracle.dequant_act_fp8(hq, sh)
    h_ref, _ = oracle.grouped_gemm(xd, off, w1, w3, w2)
    U.assert_bf16_close(h_gpu, h_ref, 2e-2, "hact from the GPU's xq")
    y_ref = np.zeros((R, H))
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi > lo:
            y_ref[lo:hi] = hd[lo:hi] @ np.asarray(w2[e], np.float64).T
    U.assert_bf16_close(U.f64(y), y_ref, 2e-2, "y from the GPU's hq")
    # end to end against the oracle's W8A8 definition
    rh, ry = oracle.grouped_gemm_w8a8(x64, off, w1, w3, w2)
    U.assert_bf16_close(h_gpu, rh, 5e-2, "hact")
    U.assert_bf16_close(U.f64(y), ry, 5e-2, "y")


def test_grouped_gemm_single_block_without_offsets(ops):
    # offsets == NULL runs one block [0, R) -- the shared-expert form
    spec = SPECS["tiny"].with_(E=1, H=512, I=256)
    for T in (3, 16, 17, 200):
        inp = synth.host_inputs(spec, T, seed=T)
        t = U.layer_tensors(inp)
        hact = torch.empty(T, spec.I, dtype=torch.bfloat16, device="cuda")
        y = torch.empty(T, spec.H, dtype=torch.bfloat16, device="cuda")
        scratch = torch.empty(ops.grouped_gemm_scratch_bytes(T, 1), dtype=torch.uint8, device="cuda")
        ops.grouped_gemm(t["x"], None, 1, spec.H, spec.I, t["w1"], t["w3"], t["w2"], hact, y, scratch)
        sync()
        w1, w3, w2 = oracle.layer_weights_f64(inp)
        rh, ry = oracle.expert_swiglu(oracle.bf16_to_f64(inp["x_bits"]), w1[0], w3[0], w2[0])
        U.assert_bf16_close(U.f64(hact), rh, what=f"hact T={T}")
        U.assert_bf16_close(U.f64(y), ry, what=f"y T={T}")


# ---------------------------------------------------------------- U
@pytest.mark.parametrize("T,K,H,shared", [(16, 2, 256, False), (1, 8, 2048, False),
                                          (333, 8, 2048, False), (64, 10, 2048, True),
                                          (7, 16, 7168, False)])
def test_unpermute(ops, T, K, H, shared):
    E = 64
    ids = synth.random_ids(T, K, E, seed=T)
    _, _, f2r = oracle.permute(ids, E)
    y_bits = synth.f32_to_bf16_bits(synth._normal(3, 1, T, (T * K, H), 1.0))
    w = np.random.default_rng(T).random((T, K)).astype(np.float32)
    sh_bits = synth.f32_to_bf16_bits(synth._normal(3, 2, T, (T, H), 1.0)) if shared else None
    g = np.random.default_rng(1).random(T).astype(np.float32) if shared else None
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    ops.unpermute(U.bf16_dev(y_bits), torch.from_numpy(f2r).cuda(), U.dev(w), T, K, H, out,
                  None if sh_bits is None else U.bf16_dev(sh_bits), U.dev(g))
    sync()
    ref = oracle.unpermute(oracle.bf16_to_f64(y_bits), f2r, w, T, K,
                           None if sh_bits is None else oracle.bf16_to_f64(sh_bits), g)
    # only the final bf16 rounding (+ fp32 sums): 2^-8 relative to the magnitude sum
    mag = oracle.unpermute(np.abs(oracle.bf16_to_f64(y_bits)), f2r, np.abs(w), T, K,
                           None if sh_bits is None else np.abs(oracle.bf16_to_f64(sh_bits)), g)
    assert (np.abs(U.f64(out) - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6 * mag + 1e-30).all()


# ---------------------------------------------------------------- whole layer
LAYER_CASES = [("tiny", {}, 16), ("tiny", {}, 1), ("qwen3_30b_a3b", {}, 1),
               ("qwen3_30b_a3b", {}, 2), ("qwen3_30b_a3b", {}, 8), ("qwen3_30b_a3b", {}, 32),
               ("qwen3_30b_a3b", {}, 256), ("gpt_oss_20b", {}, 32), ("shared_gate", {}, 4),
               ("shared_gate", {}, 64), ("shared_gate", {}, 1), ("high_expert", {}, 2),
               ("high_expert", {"E": 512, "K": 9}, 2), ("high_expert", {"E": 1024}, 1),
               # few experts active: the skinny GEMM splits K (fp32 slices + finalize)
               ("tiny", {"H": 1024, "I": 512, "E": 8, "wdtype": "fp8"}, 1),
               ("tiny", {"H": 1024, "I": 512, "E": 8, "wdtype": "fp8"}, 3),
               ("tiny", {"H": 2880, "I": 1440, "E": 4}, 1),
               ("tiny", {"H": 1024, "I": 512, "E": 8, "wdtype": "mxfp4"}, 1),
               ("gpt_oss_20b", {"wdtype": "mxfp4"}, 1), ("gpt_oss_20b", {"wdtype": "mxfp4"}, 8),
               ("gpt_oss_20b", {"wdtype": "mxfp4"}, 64),
               ("gpt_oss_20b", {"act": "fp8"}, 3), ("gpt_oss_20b", {"act": "fp8"}, 64),
               ("tiny", {"H": 1024, "I": 512, "E": 8, "wdtype": "fp8", "act": "fp8"}, 40)]


def oracle_routing(spec, inp):
    x = oracle.bf16_to_f64(inp["x_bits"])
    logits = oracle.router_logits(x, inp["wg"], inp["gate_bias"])
    if spec.mode == 0:
        ids, _ = oracle.topk_softmax_renorm(logits, spec.E, spec.K)
        keys = logits[:, :spec.E]
    else:
        ids, _ = oracle.topk_sigmoid_bias(logits.astype(np.float32), inp["sel_bias"], spec.E,
                                          spec.K, spec.routed_scale)
        s = oracle.sigmoid_f32(logits.astype(np.float32)[:, :spec.E])
        keys = (s + inp["sel_bias"][None, :]).astype(np.float64)
    srt = -np.sort(-keys, axis=1)
    margin = srt[:, spec.K - 1] - srt[:, spec.K] if spec.K < spec.E else np.full(len(ids), np.inf)
    return logits, ids, margin


@pytest.mark.parametrize("name,over,T", LAYER_CASES, ids=case_id)
def test_layer(ops, name, over, T):
    spec = SPECS[name].with_(**over)
    base = synth.host_inputs(spec, T, seed=11, weights=False)
    logits, ids, margin = oracle_routing(spec, base)
    inp = synth.host_inputs(spec, T, seed=11, experts=sorted(set(ids.ravel().tolist())))
    t = U.layer_tensors(inp, inp["experts"])
    layer = ops.MoELayer(U.config_for(ops, spec, T_max=max(T, 4)), t)
    out = layer(t["x"])
    sync()
    assert int(layer.dev_status.item()) == 0
    lg = layer.view("logits", torch.float32, (T, spec.G)).cpu().numpy()
    # intermediates
    U.assert_router_close(lg.astype(np.float64), oracle.bf16_to_f64(inp["x_bits"]), inp["wg"],
                          inp["gate_bias"])
    gid = layer.view("ids", torch.int32, (T, spec.K)).cpu().numpy()
    clear = margin > 1e-4          # fp32 router vs fp64 oracle: near ties may route either way
    assert clear.mean() > 0.9
    assert np.array_equal(gid[clear], ids[clear])
    # every token, routed by the oracle on the GPU's own logits: the ids match
    # bit for bit and the outputs element by element
    res = oracle.moe_layer_from_inputs(inp, logits_override=lg.astype(np.float64))
    assert np.array_equal(gid, res["ids"])
    rel = 5e-2 if spec.wdtype == "fp8" else 2e-2
    U.assert_bf16_close(U.f64(out), res["out"], rel, "layer out")


# T > 32: one fused routing launch (top-K, chunk histograms, and in the last
# CTA the scan to offsets and the GEMM plan) and the stable scatter.  Its
# intermediates are checked bit for bit against the oracle's permute of the
# GPU's own ids and its top-K of the GPU's own logits; its completion counter
# must come back to zero, call after call, on one workspace.
PREFILL_CASES = [("tiny", {"E": 16, "K": 4}, (33, 129, 1000, 40000)),
                 ("tiny", {"E": 40, "K": 3, "mode": 1, "routed_scale": 2.5, "sel_bias_var": 0.1},
                  (64, 777)),
                 ("high_expert", {"E": 1024, "H": 256, "I": 128}, (100,)),
                 ("shared_gate", {"H": 256, "I": 128, "I_shared": 128}, (300,))]


@pytest.mark.parametrize("name,over,Ts", PREFILL_CASES, ids=case_id)
def test_layer_prefill_routing_is_exact_and_repeats(ops, name, over, Ts):
    spec = SPECS[name].with_(**over)
    inp = synth.host_inputs(spec, max(Ts), seed=41)
    t = U.layer_tensors(inp)
    layer = ops.MoELayer(U.config_for(ops, spec, T_max=max(Ts)), t)
    for T in Ts:
        x = t["x"][:T].contiguous()
        layer(x)
        sync()
        assert int(layer.dev_status.item()) == 0
        R, E, K = T * spec.K, spec.E, spec.K
        lg = layer.view("logits", torch.float32, (T, spec.G)).cpu().numpy()
        gid = layer.view("ids", torch.int32, (T, K)).cpu().numpy()
        gw = layer.view("weights", torch.float32, (T, K)).cpu().numpy()
        if spec.mode == 0:
            rid, rw = oracle.topk_softmax_renorm(lg.astype(np.float64), E, K)
        else:
            rid, rw = oracle.topk_sigmoid_bias(lg, inp["sel_bias"], E, K, spec.routed_scale)
        assert np.array_equal(gid, rid)
        assert np.allclose(gw, rw, rtol=1e-5, atol=1e-7)
        off, r2f, f2r = oracle.permute(gid, E)
        assert np.array_equal(layer.view("offsets", torch.int32, (E + 1,)).cpu().numpy(), off)
        assert np.array_equal(layer.view("row_to_flat", torch.int32, (R,)).cpu().numpy(), r2f)
        assert np.array_equal(layer.view("flat_to_row", torch.int32, (R,)).cpu().numpy(), f2r)
        wd = U.wdtype_of(ops, spec)
        want = [ops.block_variant(int(m), R, E, -1, 0, wd) for m in np.diff(off)]
        assert layer.view("block_variant", torch.int32, (E,)).cpu().numpy().tolist() == want
        sw = layer.workspace[layer.layout.sync:layer.layout.logits].view(torch.int32)
        assert int(sw.abs().sum().item()) == 0
        if T <= 1000:
            case = dict(inp)
            case["x_bits"] = inp["x_bits"][:T]
            res = oracle.moe_layer_from_inputs(case, logits_override=lg.astype(np.float64))
            rel = 5e-2 if spec.wdtype == "fp8" else 2e-2
            U.assert_bf16_close(U.f64(layer(x)), res["out"], rel, f"prefill T={T}")


@pytest.mark.parametrize("shared", [False, True])
def test_fused_routing_one_lane_holds_every_pick(ops, shared):
    # E = 512 routes by warp-wide groups inside the fused routing launches;
    # a gate bias of +20 on the 16 experts lane 0 owns (float4 rows: e with
    # (e % 128) // 4 == 0; 513-float rows with the shared gate: e % 32 == 0)
    # makes that lane supply all K = 10 picks, past its 8-entry list
    E, K = 512, 10
    e = np.arange(E)
    own = e[e % 32 == 0] if shared else e[(e % 128) // 4 == 0]
    spec = SPECS["tiny"].with_(E=E, K=K, H=256, I=128, hot_experts=tuple(int(v) for v in own),
                               hot_bias=20.0)
    if shared:
        spec = spec.with_(has_shared=True, I_shared=128)
    inp = synth.host_inputs(spec, 100, seed=5)
    t = U.layer_tensors(inp)
    layer = ops.MoELayer(U.config_for(ops, spec, T_max=100), t)
    for T in (5, 100):  # the decode launch, then the prefill launch
        layer(t["x"][:T].contiguous())
        sync()
        assert int(layer.dev_status.item()) == 0
        lg = layer.view("logits", torch.float32, (T, spec.G)).cpu().numpy()
        gid = layer.view("ids", torch.int32, (T, K)).cpu().numpy()
        gw = layer.view("weights", torch.float32, (T, K)).cpu().numpy()
        rid, rw = oracle.topk_softmax_renorm(lg.astype(np.float64), E, K)
        assert np.array_equal(gid, rid)
        assert set(np.unique(gid).tolist()) <= set(own.tolist())
        assert np.allclose(gw, rw, rtol=1e-5, atol=1e-7)
        off, r2f, f2r = oracle.permute(gid, E)
        assert np.array_equal(layer.view("offsets", torch.int32, (E + 1,)).cpu().numpy(), off)
        assert np.array_equal(layer.view("flat_to_row", torch.int32, (T * K,)).cpu().numpy(), f2r)
        sw = layer.workspace[layer.layout.sync:layer.layout.logits].view(torch.int32)
        assert int(sw.abs().sum().item()) == 0


def test_bounded_wait_runs_out_into_a_status_word(ops):
    # the fused GEMM's cross-CTA wait, on a counter nothing increments: it
    # must give up after its limit, report MOE_DEV_WAIT_TIMEOUT and leave the
    # context usable; a satisfied wait returns at once with no status
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sync()
    t0 = time.perf_counter()
    ops.bounded_wait_check(counter, 1, 20000, st)
    sync()
    assert time.perf_counter() - t0 >= 0.02
    assert int(st.item()) == ops.DEV_WAIT_TIMEOUT
    counter.fill_(7)
    st.zero_()
    ops.bounded_wait_check(counter, 7, 20000, st)
    sync()
    assert int(st.item()) == 0
    # and the library still computes on this context
    lg = synth.random_logits(64, 32, seed=3)
    ids, w, _ = run_topk(ops, lg, 32, 4, 0, 1.0, None, False)
    rid, rw = oracle.topk_softmax_renorm(lg.astype(np.float64), 32, 4)
    assert np.array_equal(ids, rid)


def test_layer_decode_path_repeats_and_leaves_sync_zero(ops):
    # T <= 32 runs the fused routing launch; its completion counter must come
    # back to zero so that the next call (same workspace) routes again
    spec = SPECS["tiny"].with_(E=16, K=4)
    inp = synth.host_inputs(spec, 32, seed=21)
    t = U.layer_tensors(inp)
    layer = ops.MoELayer(U.config_for(ops, spec, T_max=32), t)
    for T, seed in ((8, 31), (32, 32), (3, 33), (32, 34)):
        x_bits = synth.host_inputs(spec, T, seed=seed, weights=False)["x_bits"]
        out = layer(U.bf16_dev(x_bits))
        sync()
        sw = layer.workspace[layer.layout.sync:layer.layout.logits].view(torch.int32)
        assert int(sw.abs().sum().item()) == 0
        case = dict(inp)
        case["x_bits"] = x_bits
        lg = layer.view("logits", torch.float32, (T, spec.G)).cpu().numpy()
        res = oracle.moe_layer_from_inputs(case, logits_override=lg.astype(np.float64))
        assert np.array_equal(layer.view("ids", torch.int32, (T, spec.K)).cpu().numpy(),
                              res["ids"])
        U.assert_bf16_close(U.f64(out), res["out"], 2e-2, f"decode T={T}")


# The whole layer as ONE launch (MOE_DISPATCH_ONE_LAUNCH forces it wherever it
# applies: bf16 experts, T <= 16), at every shape it takes: shared expert,
# E up to 1024 (the partitioned route for E > 128 at T <= 4), both score
# modes, H not a multiple of 128, tokens sharing experts.  Routing is compared
# bit for bit on the GPU's own logits, every output element against the
# oracle; a second call on the same workspace must give the same bits and
# leave the counters at zero.
ONE_LAUNCH_CASES = [("qwen3_30b_a3b", {}, 1), ("qwen3_30b_a3b", {}, 2), ("qwen3_30b_a3b", {}, 3),
                    ("qwen3_30b_a3b", {}, 8), ("qwen3_30b_a3b", {}, 16),
                    ("shared_gate", {}, 1), ("shared_gate", {}, 4), ("shared_gate", {}, 13),
                    ("high_expert", {}, 1), ("high_expert", {"E": 512, "K": 9}, 3),
                    ("high_expert", {"E": 1024, "K": 16, "H": 1024, "I": 512}, 4),
                    ("high_expert", {"E": 1024, "K": 9, "H": 1024, "I": 512}, 11),
                    ("tiny", {}, 16), ("tiny", {"H": 2880, "I": 1440, "E": 4}, 5),
                    ("tiny", {"E": 40, "K": 3, "mode": 1, "routed_scale": 2.5,
                              "sel_bias_var": 0.1}, 7)]


@pytest.mark.parametrize("name,over,T", ONE_LAUNCH_CASES, ids=case_id)
def test_one_launch_layer(ops, name, over, T):
    check_small_batch_layer(ops, name, over, T, ops.DISPATCH_ONE_LAUNCH, "one-launch")


# The decode batches as CUDA-core matrix-vector products (moe_layer under
# MOE_DISPATCH_GEMV): bf16 and FP8 experts, with and without the shared
# expert, T = 1..4, the largest H (the token rows staged in shared memory)
GEMV_CASES = [("qwen3_30b_a3b", {}, 1), ("qwen3_30b_a3b", {}, 2), ("qwen3_30b_a3b", {}, 3),
              ("qwen3_30b_a3b", {}, 4), ("shared_gate", {}, 1), ("shared_gate", {}, 4),
              ("gpt_oss_20b", {}, 1), ("gpt_oss_20b", {}, 4),
              ("high_expert", {}, 1), ("high_expert", {"E": 512, "K": 9}, 4),
              ("tiny", {}, 3), ("tiny", {"H": 2880, "I": 1440, "E": 4, "wdtype": "fp8"}, 2),
              ("tiny", {"E": 40, "K": 3, "mode": 1, "routed_scale": 2.5,
                        "sel_bias_var": 0.1}, 4),
              # more than 128 experts: the G1 CTAs' sliced routing with 8, 4
              # and 2 slices per token (T = 1, 2, 3), slices past E
              ("shared_gate", {}, 2), ("shared_gate", {}, 3), ("high_expert", {}, 2),
              ("tiny", {"E": 300, "K": 5}, 2),
              ("tiny", {"E": 257, "K": 7, "mode": 1, "routed_scale": 2.5,
                        "sel_bias_var": 0.1}, 3),
              # MXFP4 rows (e2m1 decoded exactly, a scale byte per 32 weights)
              ("gpt_oss_20b", {"wdtype": "mxfp4"}, 1), ("gpt_oss_20b", {"wdtype": "mxfp4"}, 2),
              ("tiny", {"H": 160, "I": 96, "E": 5, "wdtype": "mxfp4"}, 4),
              ("shared_gate", {"wdtype": "mxfp4"}, 1)]


@pytest.mark.parametrize("name,over,T", GEMV_CASES, ids=case_id)
def test_gemv_decode_layer(ops, name, over, T):
    check_small_batch_layer(ops, name, over, T, ops.DISPATCH_GEMV, "gemv")


# the matrix-vector decode path and the tensor-core path on the same inputs:
# the routing agrees bit for bit; with bf16 or MXFP4 weights (e2m1 times
# 2^(byte - 127) is exact in bf16) both read the same weight values, so hact,
# y and the output agree to the order of the fp32 sums (two bf16 steps).
# FP8 weights: the tensor-core converter rounds each code * block scale to
# bf16 for the MMA, the matrix-vector path keeps it in fp32 -- there the two
# agree to the oracle's FP8 tolerance.
GEMV_VS_TC_CASES = [("qwen3_30b_a3b", {}, 1), ("qwen3_30b_a3b", {}, 2),
                    ("gpt_oss_20b", {}, 1), ("gpt_oss_20b", {"wdtype": "mxfp4"}, 1),
                    ("gpt_oss_20b", {"wdtype": "mxfp4"}, 2), ("shared_gate", {}, 1),
                    ("high_expert", {}, 2)]


@pytest.mark.parametrize("name,over,T", GEMV_VS_TC_CASES, ids=case_id)
def test_gemv_path_matches_tensor_core_path(ops, name, over, T):
    spec = SPECS[name].with_(**over)
    base = synth.host_inputs(spec, T, seed=29, weights=False)
    _, ids, _ = oracle_routing(spec, base)
    inp = synth.host_inputs(spec, T, seed=29, experts=sorted(set(ids.ravel().tolist())))
    t = U.layer_tensors(inp, inp["experts"])
    E, K, R = spec.E, spec.K, T * spec.K
    got = {}
    for tag, disp in (("gemv", ops.DISPATCH_GEMV), ("tensor", ops.DISPATCH_GLOBAL_AVG)):
        layer = ops.MoELayer(U.config_for(ops, spec, T_max=max(T, 4), dispatch=disp), t)
        out = layer(t["x"])
        sync()
        assert int(layer.dev_status.item()) == 0
        got[tag] = {"ids": layer.view("ids", torch.int32, (T, K)).cpu().numpy(),
                    "r2f": layer.view("row_to_flat", torch.int32, (R,)).cpu().numpy(),
                    "hact": U.f64(layer.view("hact", torch.bfloat16, (R, spec.I))),
                    "y": U.f64(layer.view("y", torch.bfloat16, (R, spec.H))),
                    "out": U.f64(out)}
        del layer
    g, c = got["gemv"], got["tensor"]
    assert np.array_equal(g["ids"], c["ids"]) and np.array_equal(g["r2f"], c["r2f"])
    rel = 5e-2 if spec.wdtype == "fp8" else 8e-3
    for k in ("hact", "y", "out"):
        U.assert_bf16_close(g[k], c[k], rel, f"gemv vs tensor cores {k}")


def check_small_batch_layer(ops, name, over, T, dispatch, tag):
    spec = SPECS[name].with_(**over)
    base = synth.host_inputs(spec, T, seed=17, weights=False)
    _, ids, _ = oracle_routing(spec, base)
    inp = synth.host_inputs(spec, T, seed=17, experts=sorted(set(ids.ravel().tolist())))
    t = U.layer_tensors(inp, inp["experts"])
    layer = ops.MoELayer(U.config_for(ops, spec, T_max=max(T, 4), dispatch=dispatch), t)
    out = layer(t["x"])
    sync()
    assert int(layer.dev_status.item()) == 0
    E, K, R = spec.E, spec.K, T * spec.K
    lg = layer.view("logits", torch.float32, (T, spec.G)).cpu().numpy()
    U.assert_router_close(lg.astype(np.float64), oracle.bf16_to_f64(inp["x_bits"]), inp["wg"],
                          inp["gate_bias"])
    gid = layer.view("ids", torch.int32, (T, K)).cpu().numpy()
    gw = layer.view("weights", torch.float32, (T, K)).cpu().numpy()
    if spec.mode == 0:
        rid, rw = oracle.topk_softmax_renorm(lg.astype(np.float64), E, K)
    else:
        rid, rw = oracle.topk_sigmoid_bias(lg, inp["sel_bias"], E, K, spec.routed_scale)
    assert np.array_equal(gid, rid)
    U.assert_weights_close(gw, rw)
    off, r2f, f2r = oracle.permute(gid, E)
    assert np.array_equal(layer.view("offsets", torch.int32, (E + 1,)).cpu().numpy(), off)
    assert np.array_equal(layer.view("row_to_flat", torch.int32, (R,)).cpu().numpy(), r2f)
    assert np.array_equal(layer.view("flat_to_row", torch.int32, (R,)).cpu().numpy(), f2r)
    want = [ops.block_variant(int(m), R, E, -1, 0, U.wdtype_of(ops, spec)) for m in np.diff(off)]
    assert layer.view("block_variant", torch.int32, (E,)).cpu().numpy().tolist() == want
    res = oracle.moe_layer_from_inputs(inp, logits_override=lg.astype(np.float64))
    rel = 5e-2 if spec.wdtype == "fp8" else 2e-2
    U.assert_bf16_close(U.f64(layer.view("hact", torch.bfloat16, (R, spec.I))), res["hact"],
                        rel, f"{tag} hact")
    U.assert_bf16_close(U.f64(layer.view("y", torch.bfloat16, (R, spec.H))), res["y"], rel,
                        f"{tag} y")
    U.assert_bf16_close(U.f64(out), res["out"], rel, f"{tag} out")
    if spec.has_shared:
        U.assert_bf16_close(U.f64(layer.view("shared_y", torch.bfloat16, (T, spec.H))),
                            res["shared_y"], 2e-2, f"{tag} shared_y")
    again = layer(t["x"])
    sync()
    assert torch.equal(again.view(torch.int16), out.view(torch.int16))
    sw = layer.workspace[layer.layout.sync:layer.layout.logits].view(torch.int32)
    assert int(sw.abs().sum().item()) == 0
