"""Brute-force pins: pure-Python loops over lists, for tiny inputs only.

Written independently of ``oracle/`` (no numpy linear algebra, no shared
helpers) so that a mistake in the oracle's vectorised code cannot hide behind
the same mistake here.
"""
import math
import struct


def router(x, wg, bias=None):
    T, H, G = len(x), len(x[0]), len(wg)
    out = []
    for t in range(T):
        row = []
        for g in range(G):
            s = 0.0
            for h in range(H):
                s += x[t][h] * wg[g][h]
            if bias is not None:
                s += bias[g]
            row.append(s)
        out.append(row)
    return out


def topk_order(keys, K):
    """Indices of the K largest keys; equal keys -> lower index first."""
    return sorted(range(len(keys)), key=lambda e: (-keys[e], e))[:K]


def softmax_renorm_row(logits_row, E, K):
    sel = topk_order(list(logits_row[:E]), K)
    m = max(logits_row[e] for e in sel)
    p = [math.exp(logits_row[e] - m) for e in sel]
    s = sum(p)
    return sel, [v / s for v in p]


def sigmoid(v):
    return 1.0 / (1.0 + math.exp(-v))


def sigmoid_bias_row(logits_row, bias, E, K, scale):
    s = [sigmoid(logits_row[e]) for e in range(E)]
    keys = [s[e] + bias[e] for e in range(E)]
    sel = topk_order(keys, K)
    tot = sum(s[e] for e in sel)
    return sel, [scale * s[e] / tot for e in sel]


def permute(flat_ids, E):
    buckets = [[] for _ in range(E)]
    for f, e in enumerate(flat_ids):
        buckets[e].append(f)
    offsets = [0]
    row_to_flat = []
    for e in range(E):
        row_to_flat.extend(buckets[e])
        offsets.append(len(row_to_flat))
    flat_to_row = [0] * len(flat_ids)
    for r, f in enumerate(row_to_flat):
        flat_to_row[f] = r
    return offsets, row_to_flat, flat_to_row


def swiglu_token(a, w1, w3, w2):
    """One token through one expert with explicit loops."""
    I, H = len(w1), len(a)
    h = []
    for i in range(I):
        g = sum(a[k] * w1[i][k] for k in range(H))
        u = sum(a[k] * w3[i][k] for k in range(H))
        h.append(g / (1.0 + math.exp(-g)) * u)
    Hout = len(w2)
    return h, [sum(h[i] * w2[j][i] for i in range(I)) for j in range(Hout)]


def layer(x, wg, bias, w1, w3, w2, E, K, mode, scale=1.0, sel_bias=None, shared=None):
    """Token by token: route, run each chosen expert, weight and sum."""
    logits = router(x, wg, bias)
    out = []
    for t, xt in enumerate(x):
        if mode == 0:
            sel, w = softmax_renorm_row(logits[t], E, K)
        else:
            sel, w = sigmoid_bias_row(logits[t], sel_bias, E, K, scale)
        acc = [0.0] * len(xt)
        for e, wk in zip(sel, w):
            _, y = swiglu_token(xt, w1[e], w3[e], w2[e])
            for j in range(len(acc)):
                acc[j] += wk * y[j]
        if shared is not None:
            g = sigmoid(logits[t][E])
            _, ys = swiglu_token(xt, *shared)
            for j in range(len(acc)):
                acc[j] += g * ys[j]
        out.append(acc)
    return out


# ---------------------------------------------------------------- W8A8
def _f32(v):
    """Nearest float32 (a correctly rounded float32 operation is the double
    result rounded once: 53 >= 2 * 24 + 2 bits)."""
    return struct.unpack("<f", struct.pack("<f", v))[0]


def e4m3_decode(code):
    """OCP e4m3 ("fn"): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits;
    exponent field 0 is subnormal m * 2^-9; S.1111.111 is NaN."""
    s = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 7
    return s * (m * 2.0 ** -9 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7))


def e4m3_nearest(v):
    """Nearest finite e4m3 code (ties: even code), saturating at 448."""
    best = None
    for c in range(0x7F):  # the non-negative finite codes, 0 .. 448
        d = abs(abs(v) - e4m3_decode(c))
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    code = best[1]
    if abs(v) >= 448.0:
        code = 0x7E
    return code | (0x80 if math.copysign(1.0, v) < 0 else 0)


def quant_rows(a, block=128):
    """[R][C] floats -> (codes, scales) per row and block of columns; the
    scale and the scaled value are float32 operations."""
    codes, scales = [], []
    for row in a:
        crow, srow = [], []
        for b0 in range(0, len(row), block):
            blk = [_f32(v) for v in row[b0:b0 + block]]
            amax = max(abs(v) for v in blk)
            s = _f32(amax / 448.0)
            srow.append(s)
            crow += [0 if s == 0 else e4m3_nearest(_f32(v / s)) for v in blk]
        codes.append(crow)
        scales.append(srow)
    return codes, scales


def dequant_rows(codes, scales, block=128):
    return [[e4m3_decode(c) * srow[j // block] for j, c in enumerate(crow)]
            for crow, srow in zip(codes, scales)]


def bf16_nearest(v):
    """float64 -> float32 -> bf16 (nearest even) as a float."""
    b = struct.unpack("<I", struct.pack("<f", v))[0]
    b = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16
    return struct.unpack("<f", struct.pack("<I", b & 0xFFFFFFFF))[0]


def grouped_gemm_w8a8(xp, offsets, w1, w3, w2):
    """Per expert block: quantised x, SwiGLU, hact stored bf16, quantised
    hact, second GEMM -- loops over lists."""
    xd = dequant_rows(*quant_rows(xp))
    R, I, H = len(xp), len(w1[0]), len(w2[0])
    hact = [[0.0] * I for _ in range(R)]
    for e in range(len(offsets) - 1):
        for r in range(offsets[e], offsets[e + 1]):
            for i in range(I):
                g = sum(xd[r][h] * w1[e][i][h] for h in range(len(xd[r])))
                u = sum(xd[r][h] * w3[e][i][h] for h in range(len(xd[r])))
                hact[r][i] = bf16_nearest(g / (1.0 + math.exp(-g)) * u)
    hd = dequant_rows(*quant_rows(hact))
    y = [[0.0] * H for _ in range(R)]
    for e in range(len(offsets) - 1):
        for r in range(offsets[e], offsets[e + 1]):
            for h in range(H):
                y[r][h] = sum(hd[r][i] * w2[e][h][i] for i in range(I))
    return hact, y
