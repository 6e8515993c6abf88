"""Plain fp64 CPU oracle for the DIFF V1 and V2 backward passes (test infrastructure only).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: imported by ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs, never by the product.

The pages state the forward and report trained models, but give no backward.
The gradients here are the chain rule applied, step by step and in the
forward's own order reversed, to the operator the forward oracle computes for
one (batch, head):

    A_r = softmax(Q_r K_r^T * c)            (c = 1/sqrt d, causal or not)
    O_r = A_r V,   O = O_1 - lambda O_2
    y   = (1 - lambda_init) gamma * O / rms(O),   rms(O) = sqrt(mean_c O^2 + eps)

Given dy (the gradient of a loss with respect to y), with m = 1 - lambda_init
and Oh = O / rms(O) per row:

    g      = m gamma * dy
    dO     = (g - Oh * mean_c(g * Oh)) / rms(O)             RMSNorm
    dgamma = sum over rows of m Oh * dy
    dV     = A_1^T dO - lambda A_2^T dO
    dA_1   = dO V^T,   dA_2 = -lambda dO V^T
    dlambda = -sum(dO * O_2)
    dS_r   = A_r * (dA_r - rowsum(A_r * dA_r))              softmax
    dQ_r   = c dS_r K_r,   dK_r = c dS_r^T Q_r

Maps are built explicitly (n x n per head); meant for the sizes the tests use.
Pinned (tests/test_oracle_backward.py) to PyTorch autograd through library
routines (scaled_dot_product_attention, rms_norm) in fp64 and to central finite
differences of the forward oracle.
"""

from __future__ import annotations

import math

import numpy as np

from .diffattn_oracle import DEFAULT_EPS, _f64, attention_map


def diff_attn_v1_backward(q1, q2, k1, k2, v, lam: float, lam_init: float, gamma, eps: float,
                          causal: bool, dy) -> dict:
    """Gradients of the multi-head DIFF V1 forward (BSHD) with respect to every input.

    q*, k*: [B, n, H, d]; v, dy: [B, n, H, 2d]; gamma: [2d] or None (ones);
    one lambda shared by all heads.  Returns a dict of fp64 arrays: dq1, dq2,
    dk1, dk2 [B, n, H, d]; dv [B, n, H, 2d]; dlam (a float); dgamma [2d].
    """
    q1, q2, k1, k2, v, dy = (_f64(a) for a in (q1, q2, k1, k2, v, dy))
    B, n, H, d = q1.shape
    if v.shape != (B, n, H, 2 * d) or dy.shape != v.shape:
        raise ValueError("need q, k [B, n, H, d] and v, dy [B, n, H, 2d]")
    dv_w = 2 * d
    gam = np.ones(dv_w) if gamma is None else _f64(gamma).reshape(-1)
    m = 1.0 - lam_init
    c = 1.0 / math.sqrt(d)
    out = {name: np.zeros_like(q1) for name in ("dq1", "dq2", "dk1", "dk2")}
    out["dv"] = np.zeros_like(v)
    dlam = 0.0
    dgamma = np.zeros(dv_w)
    for b in range(B):
        for h in range(H):
            Q1, Q2, K1, K2, V, dY = (t[b, :, h] for t in (q1, q2, k1, k2, v, dy))
            # forward, kept for the backward
            A1 = attention_map(Q1, K1, c, causal)
            A2 = attention_map(Q2, K2, c, causal)
            O1, O2 = A1 @ V, A2 @ V
            O = O1 - lam * O2
            r = np.sqrt(np.mean(O * O, axis=-1, keepdims=True) + eps)
            Oh = O / r
            # RMSNorm x (1 - lambda_init) x gamma
            g = m * gam * dY
            dO = (g - Oh * np.mean(g * Oh, axis=-1, keepdims=True)) / r
            dgamma += np.sum(m * Oh * dY, axis=0)
            # O = (A1 - lambda A2) V
            out["dv"][b, :, h] = A1.T @ dO - lam * (A2.T @ dO)
            dA1 = dO @ V.T
            dA2 = -lam * (dO @ V.T)
            dlam += -float(np.sum(dO * O2))
            # softmax rows
            dS1 = A1 * (dA1 - np.sum(A1 * dA1, axis=-1, keepdims=True))
            dS2 = A2 * (dA2 - np.sum(A2 * dA2, axis=-1, keepdims=True))
            # S_r = c Q_r K_r^T
            out["dq1"][b, :, h] = c * (dS1 @ K1)
            out["dq2"][b, :, h] = c * (dS2 @ K2)
            out["dk1"][b, :, h] = c * (dS1.T @ Q1)
            out["dk2"][b, :, h] = c * (dS2.T @ Q2)
    out["dlam"] = dlam
    out["dgamma"] = dgamma
    return out


def lambda_reparam_backward(lq1, lk1, lq2, lk2, dlam: float):
    """Gradients of lambda = exp(<lq1, lk1>) - exp(<lq2, lk2>) + lambda_init.

    d lambda / d lq1 = exp(<lq1, lk1>) lk1, / d lk1 = exp(<lq1, lk1>) lq1, and
    the second term with the opposite sign; each times dlam.  Returns
    (dlq1, dlk1, dlq2, dlk2), fp64.
    """
    lq1, lk1, lq2, lk2 = (_f64(a).reshape(-1) for a in (lq1, lk1, lq2, lk2))
    e1 = math.exp(float(lq1 @ lk1))
    e2 = math.exp(float(lq2 @ lk2))
    return dlam * e1 * lk1, dlam * e1 * lq1, -dlam * e2 * lk2, -dlam * e2 * lq2




def diff_attn_v2_backward(q, k, v, lam_logits, causal: bool, dy, scale=None) -> dict:
    """Gradients of the DIFF V2 forward (oracle.diff_attn_v2) with respect to q, k, v and the logits.

    q: [B, n, Hq, d]; k, v: [B, n, Hkv, d]; lam_logits, and the returned
    dlogits: [B, n, Hq/2] (one logit per token and pair); dy: [B, n, Hq/2, d].
    Per pair g of query heads 2g, 2g + 1 over KV head kv = 2g / (Hq/Hkv), with
    s = sigmoid(logit) per row, A_e, A_o the two heads' maps:

        out   = A_e V - s * A_o V          (no norm)
        dV   += A_e^T dy - A_o^T (s * dy)
        dA_e  = dy V^T,  dA_o = -s * dy V^T
        dlogit = -s (1 - s) rowsum(dy * A_o V)
        dS    = A * (dA - rowsum(A * dA)),  dq = c dS K,  dK += c dS^T q

    dK and dV sum over every query head that reads the KV head.  Returns a dict
    of fp64 arrays dq, dk, dv, dlogits.
    """
    q, k, v, dy = (_f64(a) for a in (q, k, v, dy))
    lg = _f64(lam_logits)
    B, n, Hq, d = q.shape
    Hkv = k.shape[2]
    if Hq % 2 or Hq % Hkv or (Hq // Hkv) % 2:
        raise ValueError("need Hq even and Hq/Hkv even so each pair shares a KV head")
    G, group = Hq // 2, Hq // Hkv
    if lg.shape != (B, n, G) or dy.shape != (B, n, G, d):
        raise ValueError("need lam_logits [B, n, Hq/2] and dy [B, n, Hq/2, d]")
    c = 1.0 / math.sqrt(d) if scale is None else scale
    out = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v), "dlogits": np.zeros_like(lg)}
    for b in range(B):
        for g in range(G):
            he, ho = 2 * g, 2 * g + 1
            kv = he // group
            K, V, dY = k[b, :, kv], v[b, :, kv], dy[b, :, g]
            s = 1.0 / (1.0 + np.exp(-lg[b, :, g]))[:, None]  # [n, 1]
            Ae = attention_map(q[b, :, he], K, c, causal)
            Ao = attention_map(q[b, :, ho], K, c, causal)
            Oo = Ao @ V
            out["dv"][b, :, kv] += Ae.T @ dY - Ao.T @ (s * dY)
            dAe = dY @ V.T
            dAo = -s * (dY @ V.T)
            out["dlogits"][b, :, g] = -(s * (1.0 - s))[:, 0] * np.sum(dY * Oo, axis=-1)
            dSe = Ae * (dAe - np.sum(Ae * dAe, axis=-1, keepdims=True))
            dSo = Ao * (dAo - np.sum(Ao * dAo, axis=-1, keepdims=True))
            out["dq"][b, :, he] = c * (dSe @ K)
            out["dq"][b, :, ho] = c * (dSo @ K)
            out["dk"][b, :, kv] += c * (dSe.T @ q[b, :, he] + dSo.T @ q[b, :, ho])
    return out


__all__ = ["diff_attn_v1_backward", "diff_attn_v2_backward", "lambda_reparam_backward", "DEFAULT_EPS"]
