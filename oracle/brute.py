"""Brute-force scalar loops for tiny inputs (test infrastructure only).

A second, independent statement of the same definitions as
``diffattn_oracle.py``: pure Python loops over scalars with ``math.exp`` and
``math.sqrt``, no NumPy arithmetic, no matrix products, no broadcasting.  It
exists to pin the blocked oracle's indexing (head, token, channel, the causal
boundary, the even/odd head pairing) on inputs of a few tokens.
"""

from __future__ import annotations

import math


def _get(a, *idx):
    x = a
    for i in idx:
        x = x[i]
    return float(x)


def _softmax_weights(qrow, krows, scale, visible):
    """Weights of one query row over the visible keys (others get weight 0)."""
    scores = []
    for j, kr in enumerate(krows):
        if visible(j):
            scores.append(scale * sum(qc * kc for qc, kc in zip(qrow, kr)))
        else:
            scores.append(None)
    top = max(s for s in scores if s is not None)
    ex = [0.0 if s is None else math.exp(s - top) for s in scores]
    z = sum(ex)
    return [e / z for e in ex]


def brute_v1(q1, q2, k1, k2, v, lam, lam_init, gamma=None, eps=1e-5, causal=True):
    """DIFF V1 with per-head RMSNorm; inputs indexable as [b][t][h][c].

    Returns nested lists y[b][t][h][c].
    """
    B, n, H, d = len(q1), len(q1[0]), len(q1[0][0]), len(q1[0][0][0])
    dv = 2 * d
    scale = 1.0 / math.sqrt(d)
    y = []
    for b in range(B):
        yb = []
        for i in range(n):
            yi = []
            for h in range(H):
                def row(a, t):
                    return [_get(a, b, t, h, c) for c in range(d)]
                vis = (lambda j: j <= i) if causal else (lambda j: True)
                w1 = _softmax_weights(row(q1, i), [row(k1, j) for j in range(n)], scale, vis)
                w2 = _softmax_weights(row(q2, i), [row(k2, j) for j in range(n)], scale, vis)
                o = []
                for c in range(dv):
                    acc = 0.0
                    for j in range(n):
                        acc += (w1[j] - lam * w2[j]) * _get(v, b, j, h, c)
                    o.append(acc)
                ms = sum(x * x for x in o) / dv
                inv = 1.0 / math.sqrt(ms + eps)
                g = [1.0] * dv if gamma is None else [float(x) for x in gamma]
                yi.append([(1.0 - lam_init) * g[c] * o[c] * inv for c in range(dv)])
            yb.append(yi)
        y.append(yb)
    return y


def brute_v2(q, k, v, lam_logits, causal=True, scale=None):
    """DIFF V2: out[b][t][g][c] = attn_{2g} - sigmoid(logit[b][t][g]) * attn_{2g+1}."""
    B, n, Hq, d = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    Hkv = len(k[0][0])
    group = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = []
    for b in range(B):
        ob = []
        for i in range(n):
            oi = []
            vis = (lambda j: j <= i) if causal else (lambda j: True)
            for g in range(Hq // 2):
                heads = (2 * g, 2 * g + 1)
                attn = []
                for hq in heads:
                    kv = hq // group
                    qrow = [_get(q, b, i, hq, c) for c in range(d)]
                    krows = [[_get(k, b, j, kv, c) for c in range(d)] for j in range(n)]
                    w = _softmax_weights(qrow, krows, scale, vis)
                    attn.append([sum(w[j] * _get(v, b, j, kv, c) for j in range(n)) for c in range(d)])
                sig = 1.0 / (1.0 + math.exp(-_get(lam_logits, b, i, g)))
                oi.append([attn[0][c] - sig * attn[1][c] for c in range(d)])
            ob.append(oi)
        out.append(ob)
    return out


def brute_v1_decode(q1, q2, k1, k2, v, lam, lam_init, gamma=None, eps=1e-5, lens=None):
    """DIFF V1 decode: q[b][h][c] over the cache k[b][j][h][c], v[b][j][h][c], keys j < lens[b].

    Returns nested lists y[b][h][c] (all zeros where no key is visible).
    """
    B, n, H = len(k1), len(k1[0]), len(k1[0][0])
    d = len(k1[0][0][0])
    dv = len(v[0][0][0])
    scale = 1.0 / math.sqrt(d)
    y = []
    for b in range(B):
        L = n if lens is None else int(lens[b])
        yb = []
        for h in range(H):
            if L == 0:
                yb.append([0.0] * dv)
                continue
            q1r = [_get(q1, b, h, c) for c in range(d)]
            q2r = [_get(q2, b, h, c) for c in range(d)]
            k1r = [[_get(k1, b, j, h, c) for c in range(d)] for j in range(L)]
            k2r = [[_get(k2, b, j, h, c) for c in range(d)] for j in range(L)]
            w1 = _softmax_weights(q1r, k1r, scale, lambda j: True)
            w2 = _softmax_weights(q2r, k2r, scale, lambda j: True)
            o = [sum((w1[j] - lam * w2[j]) * _get(v, b, j, h, c) for j in range(L)) for c in range(dv)]
            ms = sum(x * x for x in o) / dv
            g = [1.0] * dv if gamma is None else [float(x) for x in gamma]
            yb.append([(1.0 - lam_init) * g[c] * o[c] / math.sqrt(ms + eps) for c in range(dv)])
        y.append(yb)
    return y
