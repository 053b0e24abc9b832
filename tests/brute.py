"""Brute-force pins: pure-Python loops over lists, for tiny inputs only.

Written independently of ``oracle/`` (no numpy linear algebra, no shared
helpers) so that a mistake in the oracle's vectorised code cannot hide behind
the same mistake here.
"""
import math


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
