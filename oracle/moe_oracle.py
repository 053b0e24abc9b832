"""CPU oracle for the MoE-layer hot path -- TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 numpy restatement of what the layer computes, written
from the five pages it is built on.  Only the tests, the package's smoke check
and the benchmark's CPU-baseline / reference arm may import it.  It shares no
code, table or helper with the CUDA library (``mixture_experts_layer_07_gb300``)
and imports nothing from it; the library never imports this module.

Pages cited below (their titles, shortened):

* [dispatch]  "vLLM CPU MoE: dynamic GEMM dispatch beyond a fixed threshold"
              (vllm PR #50949) -- sections "1. gemm.h", "2. moe_fp8.cpp".
* [router]    "vLLM MiniMax-M2 MoE gate optimisation: fused FP32 kernel"
              (vllm PR #38445) -- sections "1. Python layer", "2. CUDA kernel".
* [shared]    "vLLM fused shared-expert gate GEMM path on ROCm"
              (vllm PR #54185) -- section "code analysis".
* [permute]   "vLLM MoE permute optimisation: buffer pre-allocation"
              (vllm PR #43014) -- section "1. C++ kernel level".
* [routing]   "FlashInfer MoE routing optimisation" (flashinfer PR #4152)
              -- sections "1. routing_custom.cu", "2. routing_common.cu",
              "performance".

Every function is pinned by tests in ``tests/test_oracle_pins.py`` against
brute force, closed forms and invariants; none is "parity unpinned".

Numerics: floating point is float64 throughout, computed from the exact values
of the stored inputs (bf16 and e4m3 widen exactly).  The one place that is not
float64 is the sigmoid used as a *selection key* in sigmoid+bias routing: there
the top-K indices are compared bit for bit, so the key follows one specified
float32 formula (``sigmoid_f32``), evaluated with numpy float32 element
operations, each correctly rounded.
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------
# storage formats
# ----------------------------------------------------------------------------


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 codes -> float64.  A bf16 is the upper half of an IEEE binary32, so
    the value is the binary32 whose top 16 bits are the code (exact widening,
    [router] "2. CUDA kernel": the bf16 loads are widened to fp32 in registers)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def _e4m3_value(code: int) -> float:
    """Value of one OCP FP8 E4M3 ("fn": no infinities) code: 1 sign bit, 4
    exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds the
    subnormals m * 2^-9; S.1111.111 is NaN."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * m * 2.0 ** -9
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_to_f64(codes) -> np.ndarray:
    return _E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def dequant_fp8_block(codes, scales, block: int = 128) -> np.ndarray:
    """Dequantise e4m3 codes [..., rows, cols] with one fp32 scale per
    block x block tile (the last tile of a dimension may be narrower):
    w[r, c] = e4m3(codes[r, c]) * scales[r // block, c // block]."""
    q = e4m3_to_f64(codes)
    s = np.asarray(scales, dtype=np.float64)
    rows, cols = q.shape[-2], q.shape[-1]
    s_full = np.repeat(np.repeat(s, block, axis=-2), block, axis=-1)[..., :rows, :cols]
    return q * s_full


def _e2m1_value(code: int) -> float:
    """Value of one OCP FP4 E2M1 code: 1 sign bit, 2 exponent bits with bias
    1, 1 mantissa bit; exponent field 0 holds the subnormal m * 0.5 (so the
    magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6); no infinities or NaN."""
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * m * 0.5
    return s * (1.0 + m / 2.0) * 2.0 ** (e - 1)


_E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)


def dequant_mxfp4(packed, scales, block: int = 32) -> np.ndarray:
    """Dequantise MXFP4 rows ([dispatch] introduction: the CPU MoE path serves
    FP8 and MXFP4 experts): ``packed`` [..., rows, cols / 2] bytes hold two
    E2M1 codes each, element 2i in the low nibble and 2i + 1 in the high one;
    ``scales`` [..., rows, cols / 32] are UE8M0 bytes, scale 2^(s - 127), one
    per 32 consecutive elements of a row (OCP Microscaling):
    w[r, c] = e2m1(code[r, c]) * 2^(scales[r, c // 32] - 127)."""
    b = np.asarray(packed, dtype=np.uint8)
    codes = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    codes[..., 0::2] = b & 0xF
    codes[..., 1::2] = b >> 4
    q = _E2M1_TABLE[codes]
    e = np.asarray(scales, dtype=np.float64)
    s = np.repeat(np.exp2(e - 127.0), block, axis=-1)[..., :q.shape[-1]]
    return q * s


# W8A8: activations quantised to e4m3, one fp32 scale per (row, 128 columns).
# The pages name FP8 expert weights ([dispatch] introduction) but fix no
# activation format; the W8A8 option's definition is this one (the scale and
# the scaled value are float32 operations, as the kernels compute them, so the
# codes are a function of the inputs that both sides evaluate identically).
_E4M3_POS = np.array([_e4m3_value(c) for c in range(0x7F)], dtype=np.float64)  # 0 .. 448


def e4m3_round(v) -> np.ndarray:
    """e4m3 code of the value nearest v, ties to the even code (round to
    nearest even), magnitudes above 448 (the largest finite e4m3) saturating
    to 448; the sign bit is kept (so -0 and negatives that round to zero give
    0x80)."""
    v = np.asarray(v, np.float64)
    a = np.minimum(np.abs(v), 448.0)
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 1, 0x7E)  # POS[hi] >= a
    lo = hi - 1
    d_lo = a - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - a
    code = np.where((d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0)), hi, lo)
    return (code.astype(np.uint8) | (np.signbit(v).astype(np.uint8) << 7)).astype(np.uint8)


def quantize_act_fp8(a, block: int = 128):
    """Quantise activations [R, C] per row and per `block` consecutive columns
    (the last block may be narrower): s = float32(amax) / 448 in float32 (0
    for an all-zero block), code = e4m3_round(float32(a) / s) in float32 (0
    where s = 0).  Returns (codes uint8 [R, C], s float32 [R, ceil(C/block)])."""
    a32 = np.asarray(a, np.float32)
    R, C = a32.shape
    nb = -(-C // block)
    codes = np.zeros((R, C), np.uint8)
    sc = np.zeros((R, nb), np.float32)
    for b in range(nb):
        blk = a32[:, b * block:(b + 1) * block]
        amax = np.abs(blk).max(axis=1)
        sb = (amax / np.float32(448.0)).astype(np.float32)
        safe = np.where(sb > 0, sb, np.float32(1.0)).astype(np.float32)
        scaled = (blk / safe[:, None]).astype(np.float32)
        c = e4m3_round(scaled)
        c[sb == 0] = 0
        codes[:, b * block:(b + 1) * block] = c
        sc[:, b] = sb
    return codes, sc


def dequant_act_fp8(codes, scales, block: int = 128) -> np.ndarray:
    """w[r, c] = e4m3(codes[r, c]) * scales[r, c // block] (float64, exact)."""
    q = e4m3_to_f64(codes)
    s = np.repeat(np.asarray(scales, np.float64), block, axis=1)[:, :q.shape[1]]
    return q * s


def round_bf16(v) -> np.ndarray:
    """float64 -> float32 (nearest) -> bf16 (nearest even), back as float64:
    the rounding of a float32 result stored as bf16."""
    b = np.asarray(v, np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# R: router (gate) GEMM
# ----------------------------------------------------------------------------


def router_logits(x, wg, gate_bias=None) -> np.ndarray:
    """logits[t, g] = sum_h x[t, h] * wg[g, h] (+ gate_bias[g]).

    [router] "1. Python layer": the unfused form is F.linear(x.float(), W), a
    linear map with the gate weight in (out, in) layout; the fused kernel
    computes the same product without materialising x in fp32.  [shared]
    "code analysis": with a fused shared-expert gate the weight has E+1 rows and
    row E is that gate.  ``gate_bias`` is the optional per-column router bias
    (the GPT-OSS-shaped workload biases four experts through it).
    x: float64 [T, H]; wg: float64 [G, H]."""
    out = np.asarray(x, np.float64) @ np.asarray(wg, np.float64).T
    if gate_bias is not None:
        out = out + np.asarray(gate_bias, np.float64)[None, :]
    return out


# ----------------------------------------------------------------------------
# K: top-K routing
# ----------------------------------------------------------------------------


def _order_desc_low_index(keys_row) -> np.ndarray:
    """Indices sorted by key descending; equal keys keep ascending index order
    (stable sort of the negated key; -0 and +0 compare equal)."""
    return np.argsort(-np.asarray(keys_row), kind="stable")


def topk_softmax_renorm(logits, E: int, K: int):
    """Softmax over the E routed logits, keep the top K, renormalise to sum 1.

    Selection is by raw logit (softmax is monotone, so the set is the same),
    highest first, lowest expert index first among equal logits.  The weights
    are p_k / sum_sel p, which equals the softmax taken over the K selected
    logits only.  Columns >= E (a fused shared-expert gate) are ignored.
    Returns ids int32 [T, K] and weights float64 [T, K]."""
    lg = np.asarray(logits)[:, :E]
    T = lg.shape[0]
    ids = np.empty((T, K), dtype=np.int32)
    w = np.empty((T, K), dtype=np.float64)
    for t in range(T):
        sel = _order_desc_low_index(lg[t])[:K]
        ids[t] = sel
        l = lg[t, sel].astype(np.float64)
        p = np.exp(l - l.max())
        w[t] = p / p.sum()
    return ids, w


# --- the float32 sigmoid used as a bit-exact selection key ------------------
# exp(z) by Cody-Waite range reduction z = n*ln2 + r with |r| <= ln2/2, ln2
# split into a 15-significant-bit head (so n*LN2_HI is exact for |n| < 512) and
# a float32 tail, then the degree-7 Taylor polynomial of e^r in Horner form,
# then scaling by 2^n.  Every step is one correctly rounded float32 operation
# (multiply and add kept separate, never fused).

_F = np.float32
_LOG2E = _F(1.4426950408889634)
_LN2_HI = _F(0.693145751953125)                  # 0x3F317200
_LN2_LO = _F(0.6931471805599453 - 0.693145751953125)
_TAYLOR = [_F(1.0 / f) for f in (5040.0, 720.0, 120.0, 24.0, 6.0, 2.0, 1.0, 1.0)]


def _exp_f32_reduced(z: np.ndarray) -> np.ndarray:
    """exp(z) for float32 z in [-87, 88] by the reduction above (elementwise)."""
    z = np.asarray(z, dtype=np.float32)
    n = np.rint(z * _LOG2E).astype(np.float32)          # nearest, ties to even
    r = (z - n * _LN2_HI).astype(np.float32)
    r = (r - n * _LN2_LO).astype(np.float32)
    p = np.full_like(r, _TAYLOR[0])
    for c in _TAYLOR[1:]:
        p = (p * r).astype(np.float32)
        p = (p + c).astype(np.float32)
    # 2^n built from its exponent field (n in [-126, 127], a normal number)
    two_n = ((n.astype(np.int32) + 127).astype(np.uint32) << np.uint32(23)).view(np.float32)
    return (p * two_n).astype(np.float32)


def sigmoid_f32(logits) -> np.ndarray:
    """sigma(l) = 1 / (1 + exp(-l)) in float32 by the specified formula:
    z = -l; z > 88 -> 0; z < -87 -> 1; else 1 / (1 + exp_f32(z)), with one
    correctly rounded float32 add and one correctly rounded float32 divide."""
    l = np.asarray(logits, dtype=np.float32)
    z = (-l).astype(np.float32)
    zc = np.clip(z, _F(-87.0), _F(88.0))
    e = _exp_f32_reduced(zc)
    den = (_F(1.0) + e).astype(np.float32)
    s = (_F(1.0) / den).astype(np.float32)
    s = np.where(z > _F(88.0), _F(0.0), s)
    s = np.where(z < _F(-87.0), _F(1.0), s)
    return s.astype(np.float32)


def topk_sigmoid_bias(logits_f32, sel_bias, E: int, K: int, scale: float):
    """SigmoidBias selection with ScaledSumNormalize weights ([routing]
    "performance" names the policy; the workload defines it):

      s_e   = sigmoid(l_e)                 (float32, ``sigmoid_f32``)
      key_e = s_e + bias_e                 (one float32 add)
      pick the K largest keys (lowest index first among equal keys)
      w_k   = scale * s_k / sum_{selected} s     (unbiased sigmoids, float64)

    Returns ids int32 [T, K], weights float64 [T, K]."""
    lg = np.asarray(logits_f32, dtype=np.float32)[:, :E]
    s = sigmoid_f32(lg)
    b = (np.zeros(E, np.float32) if sel_bias is None
         else np.asarray(sel_bias, dtype=np.float32))
    key = (s + b[None, :]).astype(np.float32)
    T = lg.shape[0]
    ids = np.empty((T, K), dtype=np.int32)
    w = np.empty((T, K), dtype=np.float64)
    for t in range(T):
        sel = _order_desc_low_index(key[t])[:K]
        ids[t] = sel
        ss = s[t, sel].astype(np.float64)
        w[t] = scale * ss / ss.sum()
    return ids, w


def shared_gate(logits, E: int) -> np.ndarray:
    """Shared-expert gate g[t] = sigmoid(logits[t, E]) (float64): row E of the
    fused gate weight ([shared] "code analysis", width 512 + 1)."""
    l = np.asarray(logits, dtype=np.float64)[:, E]
    return 1.0 / (1.0 + np.exp(-l))


# ----------------------------------------------------------------------------
# P: permute
# ----------------------------------------------------------------------------


def permute(ids, E: int):
    """Stable counting sort of the token replicas by expert.

    Replica f = t*K + k (expert ids[t, k]) goes to row
    offsets[e] + (number of replicas f' < f with the same expert), so each
    expert's rows form one contiguous block [offsets[e], offsets[e+1]) whose
    size is m_size = offsets[e+1] - offsets[e] ([dispatch] "2. moe_fp8.cpp").
    Returns offsets int32 [E+1], row_to_flat int32 [R], flat_to_row int32 [R]."""
    flat = np.asarray(ids, dtype=np.int64).ravel()
    counts = np.bincount(flat, minlength=E)[:E]
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    row_to_flat = np.argsort(flat, kind="stable")
    flat_to_row = np.empty_like(row_to_flat)
    flat_to_row[row_to_flat] = np.arange(flat.size)
    return (offsets.astype(np.int32), row_to_flat.astype(np.int32),
            flat_to_row.astype(np.int32))


def gather_rows(x, row_to_flat, K: int) -> np.ndarray:
    """Xp[row] = x[row_to_flat[row] // K]: the permuted activation copy."""
    return np.asarray(x)[np.asarray(row_to_flat) // K]


# ----------------------------------------------------------------------------
# G1 / G2: grouped SwiGLU expert GEMM
# ----------------------------------------------------------------------------


def silu(z):
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def expert_swiglu(a, w1, w3, w2):
    """One expert: h = silu(a W1^T) * (a W3^T);  y = h W2^T  (float64, no
    intermediate rounding).  a [m, H]; w1, w3 [I, H]; w2 [H, I]."""
    a = np.asarray(a, np.float64)
    h = silu(a @ np.asarray(w1, np.float64).T) * (a @ np.asarray(w3, np.float64).T)
    return h, h @ np.asarray(w2, np.float64).T


def grouped_gemm(xp, offsets, w1, w3, w2):
    """Run every expert block [offsets[e], offsets[e+1]) through its own SwiGLU
    MLP.  A block with m_size == 0 is skipped ([dispatch] "2. moe_fp8.cpp").
    Which kernel variant the GPU picks for a block (from its m_size) does not
    change the mathematics, so the oracle has a single path.
    Returns hact float64 [R, I] and y float64 [R, H]."""
    xp = np.asarray(xp, np.float64)
    R = xp.shape[0]
    E = len(offsets) - 1
    I, H = w1.shape[1], w1.shape[2]
    hact = np.zeros((R, I))
    y = np.zeros((R, H))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        hact[lo:hi], y[lo:hi] = expert_swiglu(xp[lo:hi], w1[e], w3[e], w2[e])
    return hact, y


def grouped_gemm_w8a8(xp, offsets, w1, w3, w2):
    """``grouped_gemm`` with both GEMMs' activations quantised (W8A8): the
    expert input xp -> quantize_act_fp8 -> dequantised x~; h = silu(x~ W1^T) *
    (x~ W3^T); hact = h stored as bf16 (round_bf16); hact -> quantize_act_fp8
    -> h~; y = h~ W2^T.  Weights as given (the dequantised FP8 experts).
    Returns hact (the bf16 values, float64) and y float64."""
    xp = np.asarray(xp, np.float64)
    R = xp.shape[0]
    E = len(offsets) - 1
    I, H = w1.shape[1], w1.shape[2]
    xd = dequant_act_fp8(*quantize_act_fp8(xp)) if R else xp
    hact = np.zeros((R, I))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            a = xd[lo:hi]
            hact[lo:hi] = round_bf16(silu(a @ np.asarray(w1[e], np.float64).T) *
                                     (a @ np.asarray(w3[e], np.float64).T))
    hd = dequant_act_fp8(*quantize_act_fp8(hact)) if R else hact
    y = np.zeros((R, H))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            y[lo:hi] = hd[lo:hi] @ np.asarray(w2[e], np.float64).T
    return hact, y


# ----------------------------------------------------------------------------
# U: weighted unpermute / combine
# ----------------------------------------------------------------------------


def unpermute(y, flat_to_row, weights, T: int, K: int, shared_y=None, g_sh=None):
    """out[t] = sum_k w[t, k] * y[flat_to_row[t*K + k]]  (+ g_sh[t] * shared_y[t]).

    [permute] introduction: unpermute is the inverse of permute that brings the
    expert outputs back to token order and combines them."""
    y = np.asarray(y, np.float64)
    f2r = np.asarray(flat_to_row).reshape(T, K)
    w = np.asarray(weights, np.float64).reshape(T, K)
    out = np.einsum("tk,tkh->th", w, y[f2r])
    if shared_y is not None:
        out = out + np.asarray(g_sh, np.float64)[:, None] * np.asarray(shared_y, np.float64)
    return out


# ----------------------------------------------------------------------------
# the whole layer
# ----------------------------------------------------------------------------


class ExpertBank:
    """Read-only [E, rows, cols] view of stored expert weights that decodes one
    expert to float64 when it is indexed (bf16 codes widened, or e4m3 codes
    dequantised by block), so a layer with many large experts never holds all
    of them in float64 at once."""

    def __init__(self, codes, scales=None, fmt="bf16"):
        self.codes = codes
        self.scales = scales
        self.fmt = fmt
        shape = tuple(codes.shape)
        # MXFP4 rows hold two elements per byte
        self.shape = shape[:-1] + (2 * shape[-1],) if fmt == "mxfp4" else shape

    def __getitem__(self, e):
        if self.fmt == "mxfp4":
            return dequant_mxfp4(self.codes[e], self.scales[e])
        if self.scales is None:
            return bf16_to_f64(self.codes[e])
        return dequant_fp8_block(self.codes[e], self.scales[e])

    def __len__(self):
        return self.shape[0]


def layer_weights_f64(inp: dict):
    """Expert weights of an input dict (see the package's ``synth`` module) as
    three ``ExpertBank``s: W1 [E, I, H], W3 [E, I, H], W2 [E, H, I] (bf16, FP8
    or MXFP4 storage)."""
    if "w1_bits" in inp:
        return (ExpertBank(inp["w1_bits"]), ExpertBank(inp["w3_bits"]),
                ExpertBank(inp["w2_bits"]))
    if "w1_q4" in inp:
        return (ExpertBank(inp["w1_q4"], inp["s1"], "mxfp4"),
                ExpertBank(inp["w3_q4"], inp["s3"], "mxfp4"),
                ExpertBank(inp["w2_q4"], inp["s2"], "mxfp4"))
    return (ExpertBank(inp["w1_q"], inp["s1"]), ExpertBank(inp["w3_q"], inp["s3"]),
            ExpertBank(inp["w2_q"], inp["s2"]))


def moe_layer(x, wg, gate_bias, sel_bias, w1, w3, w2, *, E: int, K: int, mode: int,
              routed_scale: float = 1.0, shared=None, logits_override=None, w8a8=False):
    """The whole hot path: R -> K -> P -> G1/G2 -> U, float64.

    ``shared`` = (sw1, sw3, sw2) adds g_sh[t] * SwiGLU_shared(x[t]).
    ``logits_override`` (float32 [T, G]) replaces the router output for the
    routing step only (used to study near-tied selections).
    ``w8a8``: the routed experts' GEMMs quantise their activations
    (``grouped_gemm_w8a8``); the shared expert stays bf16.
    Returns a dict with every intermediate."""
    x = np.asarray(x, np.float64)
    T = x.shape[0]
    logits = router_logits(x, wg, gate_bias)
    lsel = logits if logits_override is None else logits_override
    if mode == 0:
        ids, w = topk_softmax_renorm(lsel, E, K)
    else:
        ids, w = topk_sigmoid_bias(np.asarray(lsel, np.float32), sel_bias, E, K, routed_scale)
    offsets, row_to_flat, flat_to_row = permute(ids, E)
    xp = gather_rows(x, row_to_flat, K)
    hact, y = (grouped_gemm_w8a8 if w8a8 else grouped_gemm)(xp, offsets, w1, w3, w2)
    sh, g = None, None
    if shared is not None:
        g = shared_gate(logits, E)
        _, sh = expert_swiglu(x, *shared)
    out = unpermute(y, flat_to_row, w, T, K, sh, g)
    return dict(logits=logits, ids=ids, weights=w, offsets=offsets, row_to_flat=row_to_flat,
                flat_to_row=flat_to_row, xp=xp, hact=hact, y=y, shared_y=sh, shared_gate=g,
                out=out)


def moe_layer_from_inputs(inp: dict, logits_override=None):
    """``moe_layer`` on a host input dict drawn by the package's ``synth``."""
    spec = inp["spec"]
    x = bf16_to_f64(inp["x_bits"])
    w1, w3, w2 = layer_weights_f64(inp)
    shared = None
    if spec.has_shared:
        shared = (bf16_to_f64(inp["sw1_bits"]), bf16_to_f64(inp["sw3_bits"]),
                  bf16_to_f64(inp["sw2_bits"]))
    return moe_layer(x, inp["wg"], inp["gate_bias"], inp["sel_bias"], w1, w3, w2,
                     E=spec.E, K=spec.K, mode=spec.mode, routed_scale=spec.routed_scale,
                     shared=shared, logits_override=logits_override,
                     w8a8=getattr(spec, "act", "bf16") == "fp8")
