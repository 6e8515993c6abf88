"""fp64 CPU oracle of the attention layer around the path: projections in, W^O out.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``.

[NEWS] "差分注意力": the input X is projected to Q_1, Q_2, K_1, K_2 and V by
the parameter matrices W^Q, W^K, W^V; with h heads each head i has its own
W^Q_i, W^K_i, W^V_i, lambda is shared by the heads of a layer, every head's
output is normalised on its own (RMSNorm with the fixed multiplier
1 - lambda_init), the heads are concatenated along the channels and
projected by W^O.  [V2] "5. 간소화된 λ 매개변수화": lambda is learned per token
and per head (a sigmoid of a logit); "GQA와의 호환성": 2h query heads over h KV
heads, pairs of adjacent query heads differenced.

Readings where the equations are missing from the pages:
  * V1: the projection X W^Q of head i is 2d wide and splits into Q_1 (first
    d columns) and Q_2 (last d); the same for K; V of head i is 2d wide.
    Weights are stored as [D, H * 2d] with head i in columns
    [i * 2d, (i + 1) * 2d) (any other fixed split is a permutation of the
    columns of W^Q, W^K).
  * V2: q = X W^Q [D, Hq * d], k = X W^K and v = X W^V [D, Hkv * d], and the
    logits of the head pairs are a projection of the token, X W^lambda
    [D, Hq / 2]; out = Concat(pairs) W^O with W^O [Hq / 2 * d, D].
  * No biases.
"""

from __future__ import annotations

import numpy as np

from .diffattn_oracle import DEFAULT_EPS, _f64, diff_attn_v1, diff_attn_v2, lambda_reparam


def diff_v1_layer(x, wq, wk, wv, wo, lq1, lk1, lq2, lk2, lam_init: float, H: int, gamma=None,
                  eps: float = DEFAULT_EPS, causal: bool = True) -> np.ndarray:
    """Multi-head DIFF V1 attention layer: projections, DiffAttn per head, per-head norm, W^O.

    x: [B, n, D]; wq, wk, wv: [D, H * 2d]; wo: [H * 2d, D].  Returns [B, n, D] (fp64).
    """
    x, wq, wk, wv, wo = (_f64(a) for a in (x, wq, wk, wv, wo))
    B, n, D = x.shape
    if wq.shape[0] != D or wq.shape[1] % (2 * H):
        raise ValueError("wq must be [D, H * 2d]")
    d = wq.shape[1] // (2 * H)
    if wk.shape != wq.shape or wv.shape != wq.shape or wo.shape != (H * 2 * d, D):
        raise ValueError("need wk, wv [D, H * 2d] and wo [H * 2d, D]")
    q = (x @ wq).reshape(B, n, H, 2 * d)
    k = (x @ wk).reshape(B, n, H, 2 * d)
    v = (x @ wv).reshape(B, n, H, 2 * d)
    lam = lambda_reparam(lq1, lk1, lq2, lk2, lam_init)
    y = diff_attn_v1(q[..., :d], q[..., d:], k[..., :d], k[..., d:], v, lam, lam_init, gamma, eps, causal)
    return y.reshape(B, n, H * 2 * d) @ wo


def diff_v2_layer(x, wq, wk, wv, wl, wo, Hq: int, Hkv: int, causal: bool = True) -> np.ndarray:
    """DIFF V2 attention layer: projections (and per-token logits), GQA DiffAttn V2, W^O.

    x: [B, n, D]; wq: [D, Hq * d]; wk, wv: [D, Hkv * d]; wl: [D, Hq / 2];
    wo: [Hq / 2 * d, D].  Returns [B, n, D] (fp64).
    """
    x, wq, wk, wv, wl, wo = (_f64(a) for a in (x, wq, wk, wv, wl, wo))
    B, n, D = x.shape
    if wq.shape[0] != D or wq.shape[1] % Hq:
        raise ValueError("wq must be [D, Hq * d]")
    d = wq.shape[1] // Hq
    G = Hq // 2
    if wk.shape != (D, Hkv * d) or wv.shape != (D, Hkv * d) or wl.shape != (D, G) or wo.shape != (G * d, D):
        raise ValueError("need wk, wv [D, Hkv * d], wl [D, Hq / 2] and wo [Hq / 2 * d, D]")
    q = (x @ wq).reshape(B, n, Hq, d)
    k = (x @ wk).reshape(B, n, Hkv, d)
    v = (x @ wv).reshape(B, n, Hkv, d)
    logits = x @ wl  # [B, n, Hq / 2]
    y = diff_attn_v2(q, k, v, logits, causal)
    return y.reshape(B, n, G * d) @ wo
