"""Plain, slow fp64 CPU oracle for the multi-head differential-attention forward.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py`` (its CPU-baseline and reference legs).  Nothing on the
product path imports it, and it imports nothing from the product package.

Every function is the textbook definition written out with NumPy in float64,
with no blocking beyond "a block of query rows at a time" (so that a 65536-token
sequence never builds an n x n matrix) and no fusion: the maps are built
explicitly, subtracted, multiplied by V, then normalised.

Sources (web pages on the Differential Transformer; cited by title and section):
  [GLOSSARY]  "Differential Transformer", ultralytics.com glossary (Korean and
              Russian editions), section "How differential attention works"
              (Korean: 차등 어텐션의 작동 방식) with its worked example.
  [V2]        "Differential Transformer V2 (DIFF V2) 기술적 혁신 분석",
              neuralnode.tistory.com: sections "차등 어텐션 메커니즘의 핵심 원리"
              (the operator), "DIFF V1의 한계와 문제점" (lambda formulas, RMS
              range), "DIFF V2의 핵심 기술적 혁신" (code, sigmoid lambda, RMS
              table), "GQA와의 호환성" (even/odd head pairing).
  [SUMMARY]   milk-kwon.tistory.com summary, section "2. Differential
              Transformer 핵심 아이디어" (operator; per-head RMSNorm).
  [NEWS]      esgcw.com.cn news article, section "差分注意力" (projections,
              lambda re-parameterisation, lambda_init schedule, multi-head,
              per-head RMSNorm with the fixed (1 - lambda_init) multiplier).
  [FP8]       The OCP 8-bit floating point specification (E4M3): the byte
              format of an FP8 key cache; the [GLOSSARY] page only motivates
              low-bit attention by DIFF's smaller activation outliers.

Readings where the pages are silent or garbled:
  * scale 1/sqrt(d) with d the per-map query/key width ([GLOSSARY] code; the
    [V2] and [SUMMARY] formulas omit it, the [NEWS] equation was stripped);
  * causal mask: key j visible to query i iff j <= i (decoder-only, [NEWS]);
  * per-head RMSNorm over the 2d channels of one (token, head), eps = 1e-5 by
    default, one gamma of length 2d shared by all heads;
  * the multiplier is the constant (1 - lambda_init), not (1 - lambda);
  * DIFF V2 splits even/odd *heads* (the slice axis in the printed snippet is
    garbled); its lambda is sigmoid(logit) with one logit per (token, pair).

Parity pins: every function here is checked in ``tests/test_oracle_*.py``
against values the pages print, closed forms, invariants, library routines
(torch SDPA / rms_norm in fp64) and brute-force loops (``oracle/brute.py``).
No function is "parity unpinned".
"""

from __future__ import annotations

import math

import numpy as np

DEFAULT_EPS = 1e-5
ROW_BLOCK = 128


def _f64(x) -> np.ndarray:
    """Exact fp64 copy of an array-like (bf16/fp32 torch tensors included)."""
    if hasattr(x, "detach"):  # a torch tensor: upcast exactly on the host
        x = x.detach().to("cpu")
        if str(x.dtype) in ("torch.bfloat16", "torch.float16"):
            x = x.float()
        x = x.double().numpy()
    return np.asarray(x, dtype=np.float64)


def lambda_init(layer_index: int) -> float:
    """lambda_init for 1-based layer index l: 0.8 - 0.6 * exp(-0.3 * (l - 1)).

    [NEWS] section "差分注意力" (lambda_init paragraph, l in [1, L]);
    [V2] section "DIFF V1의 한계와 문제점" (fourth limit);
    [GLOSSARY] prose after the worked example.
    """
    if int(layer_index) != layer_index or layer_index < 1:
        raise ValueError("layer_index is 1-based and must be >= 1")
    return 0.8 - 0.6 * math.exp(-0.3 * (layer_index - 1))


def lambda_reparam(lq1, lk1, lq2, lk2, lam_init: float) -> float:
    """lambda = exp(<lq1, lk1>) - exp(<lq2, lk2>) + lambda_init.

    The sums over products in the printed formula are inner products of the
    four learnable vectors.  [V2] "DIFF V1의 한계와 문제점" and section 5 of
    "DIFF V2의 핵심 기술적 혁신"; [NEWS] "差分注意力" (re-parameterisation).
    """
    lq1, lk1, lq2, lk2 = (_f64(a).reshape(-1) for a in (lq1, lk1, lq2, lk2))
    if not (lq1.shape == lk1.shape == lq2.shape == lk2.shape):
        raise ValueError("the four lambda vectors must have the same length")
    return float(math.exp(float(np.dot(lq1, lk1))) - math.exp(float(np.dot(lq2, lk2))) + lam_init)


def sigmoid(x):
    """Logistic function 1 / (1 + exp(-x)), fp64 ([V2] section 5, sigmoid lambda)."""
    x = _f64(x)
    return 1.0 / (1.0 + np.exp(-x))


def softmax_rows(s: np.ndarray) -> np.ndarray:
    """Row softmax: subtract the row maximum, exponentiate, divide by the row sum."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def _rows(rows, n):
    if rows is None:
        return np.arange(n)
    rows = np.asarray(rows, dtype=np.int64).reshape(-1)
    if rows.size and (rows.min() < 0 or rows.max() >= n):
        raise IndexError("query row out of range")
    return rows


def attention_map(q, k, scale: float, causal: bool, rows=None) -> np.ndarray:
    """One softmax attention map softmax(Q K^T * scale) for the given query rows.

    q: [n_q, d], k: [n_k, d] (one head).  Returns [len(rows), n_k].  With
    ``causal`` query i sees key j iff j <= i.  [GLOSSARY] worked example;
    [V2] "Attention(Q, K, V) = Softmax(QK^T / sqrt d) V".
    """
    q = _f64(q)
    k = _f64(k)
    rows = _rows(rows, q.shape[0])
    s = (q[rows] @ k.T) * scale
    if causal:
        j = np.arange(k.shape[0])[None, :]
        s = np.where(j <= rows[:, None], s, -np.inf)
    return softmax_rows(s)


def difference_map(q1, k1, q2, k2, lam: float, causal: bool, rows=None, scale=None) -> np.ndarray:
    """The differential map softmax(Q1 K1^T/sqrt d) - lambda * softmax(Q2 K2^T/sqrt d).

    [GLOSSARY] "(map1 - lambda x map2) x V" and its code; [V2] DiffAttn formula;
    [SUMMARY] operator; d is the per-map query/key width.
    """
    d = _f64(q1).shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    a1 = attention_map(q1, k1, scale, causal, rows)
    a2 = attention_map(q2, k2, scale, causal, rows)
    return a1 - lam * a2


def diff_attn_head(q1, q2, k1, k2, v, lam: float, causal: bool, rows=None, scale=None) -> np.ndarray:
    """Pre-norm output O = (A1 - lambda A2) V of one head, row block by row block.

    q*, k*: [n, d]; v: [n, 2d].  Returns [len(rows), 2d].
    """
    q1, q2, k1, k2, v = (_f64(a) for a in (q1, q2, k1, k2, v))
    rows = _rows(rows, q1.shape[0])
    out = np.empty((rows.size, v.shape[1]), dtype=np.float64)
    for s in range(0, rows.size, ROW_BLOCK):
        blk = rows[s:s + ROW_BLOCK]
        dmap = difference_map(q1, k1, q2, k2, lam, causal, blk, scale)
        out[s:s + blk.size] = dmap @ v
    return out


def head_rmsnorm(o, gamma, eps: float, lam_init: float) -> np.ndarray:
    """Per-head RMSNorm scaled by the fixed multiplier (1 - lambda_init).

    y = (1 - lambda_init) * gamma * o / sqrt(mean(o^2) + eps), the mean taken
    over the 2d channels of one (token, head).  [NEWS] "差分注意力" (LN applies
    RMSNorm to each head; fixed multiplier (1 - lambda_init)); [SUMMARY]
    "Multi-head Differential Attention"; [GLOSSARY] prose after the example.
    """
    o = _f64(o)
    g = np.ones(o.shape[-1]) if gamma is None else _f64(gamma).reshape(-1)
    ms = np.mean(o * o, axis=-1, keepdims=True)
    return (1.0 - lam_init) * g * o / np.sqrt(ms + eps)


def diff_attn_v1(q1, q2, k1, k2, v, lam: float, lam_init: float, gamma=None,
                 eps: float = DEFAULT_EPS, causal: bool = True, rows=None) -> np.ndarray:
    """Multi-head DIFF V1 forward in BSHD layout.

    q1, q2, k1, k2: [B, n, H, d]; v: [B, n, H, 2d]; one lambda shared by all
    heads ([NEWS] "the scalar lambda is shared between heads of a layer").
    Returns y: [B, len(rows), H, 2d] (fp64).
    """
    q1, q2, k1, k2, v = (_f64(a) for a in (q1, q2, k1, k2, v))
    B, n, H, d = q1.shape
    if v.shape != (B, n, H, 2 * d):
        raise ValueError("v must be [B, n, H, 2d]")
    rows = _rows(rows, n)
    y = np.empty((B, rows.size, H, 2 * d), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            o = diff_attn_head(q1[b, :, h], q2[b, :, h], k1[b, :, h], k2[b, :, h], v[b, :, h],
                               lam, causal, rows)
            y[b, :, h] = head_rmsnorm(o, gamma, eps, lam_init)
    return y


def diff_attn_v1_decode(q1, q2, k1, k2, v, lam: float, lam_init: float, gamma=None,
                        eps: float = DEFAULT_EPS, lens=None) -> np.ndarray:
    """DIFF V1 for one new token per sequence over a key/value cache (decode).

    q1, q2: [B, H, d], the new token's queries; k1, k2: [B, n, H, d] and v:
    [B, n, H, 2d], the cache (the new token's own keys included); lens: [B]
    keys visible to sequence b (keys j < lens[b]), default n.  The output of a
    head is the same operator as one row of diff_attn_v1: the difference of
    two softmax maps over the visible keys times V, then the per-head RMSNorm
    with the fixed (1 - lambda_init).  Reading where the pages are silent: a
    sequence with no visible key (lens[b] = 0) gets an all-zero output.
    Returns [B, H, 2d] (fp64).
    """
    q1, q2, k1, k2, v = (_f64(a) for a in (q1, q2, k1, k2, v))
    B, n, H, d = k1.shape
    if q1.shape != (B, H, d) or q2.shape != (B, H, d) or v.shape != (B, n, H, 2 * d):
        raise ValueError("need q [B, H, d], k [B, n, H, d], v [B, n, H, 2d]")
    lens = np.full(B, n, dtype=np.int64) if lens is None else np.asarray(lens, dtype=np.int64).reshape(-1)
    if lens.shape != (B,) or lens.min(initial=0) < 0 or lens.max(initial=0) > n:
        raise ValueError("lens must be [B] with 0 <= len <= n")
    y = np.zeros((B, H, 2 * d), dtype=np.float64)
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        for h in range(H):
            o = diff_attn_head(q1[b, None, h], q2[b, None, h], k1[b, :L, h], k2[b, :L, h], v[b, :L, h],
                               lam, causal=False)
            y[b, h] = head_rmsnorm(o, gamma, eps, lam_init)[0]
    return y


def diff_attn_v2(q, k, v, lam_logits, causal: bool = True, scale=None, rows=None,
                 pairing: str = "adjacent") -> np.ndarray:
    """DIFF V2 forward: out_g = attn[2g] - sigmoid(lambda_g) * attn[2g+1].

    q: [B, n, Hq, d]; k, v: [B, n, Hkv, d] (grouped-query attention: query head
    j reads KV head j // (Hq/Hkv)).  lam_logits: [B, n, Hq/2] (one logit per
    token and head pair).  Returns [B, len(rows), Hq/2, d].  No RMSNorm.
    [V2] "2. 커스텀 커널 제거" (code), "5. 간소화된 λ 매개변수화" (sigmoid),
    "3. Softmax 크기 제약 극복" (norm removed), "GQA와의 호환성" (even/odd pairs).

    ``pairing="halves"`` is the first-half/second-half split that the GQA
    section calls wrong; it exists only so a test can show it differs.
    """
    q, k, v = (_f64(a) for a in (q, k, v))
    B, n, Hq, d = q.shape
    Hkv = k.shape[2]
    if Hq % 2 or Hq % Hkv or (Hq // Hkv) % 2:
        raise ValueError("need Hq even and Hq/Hkv even so each pair shares a KV head")
    group = Hq // Hkv
    lam_logits = _f64(lam_logits)
    if lam_logits.shape != (B, n, Hq // 2):
        raise ValueError("lam_logits must be [B, n, Hq/2]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rows = _rows(rows, n)
    out = np.empty((B, rows.size, Hq // 2, d), dtype=np.float64)
    for b in range(B):
        for g in range(Hq // 2):
            if pairing == "adjacent":
                he, ho = 2 * g, 2 * g + 1
            elif pairing == "halves":
                he, ho = g, g + Hq // 2
            else:
                raise ValueError(pairing)
            sig = sigmoid(lam_logits[b, rows, g])[:, None]
            for s in range(0, rows.size, ROW_BLOCK):
                blk = rows[s:s + ROW_BLOCK]
                ke, ko = he // group, ho // group
                oe = attention_map(q[b, :, he], k[b, :, ke], scale, causal, blk) @ v[b, :, ke]
                oo = attention_map(q[b, :, ho], k[b, :, ko], scale, causal, blk) @ v[b, :, ko]
                out[b, s:s + blk.size, g] = oe - sig[s:s + blk.size] * oo
    return out


def diff_attn_v2_decode(q, k, v, lam_logits, lens=None, scale=None) -> np.ndarray:
    """DIFF V2 for one new token per sequence over a key/value cache (decode).

    q: [B, Hq, d], the new token's query heads; k, v: [B, n, Hkv, d], the cache
    (the new token's own keys included); lam_logits: [B, Hq/2], the new
    token's logit per head pair; lens: [B] visible keys (keys j < lens[b]),
    default n.  out_g = A_{2g} - sigmoid(logit_g) A_{2g+1} over the visible
    keys, A_j reading KV head j // (Hq/Hkv): the same operator as one row of
    diff_attn_v2.  A sequence with no visible key gets zeros.
    Returns [B, Hq/2, d] (fp64).
    """
    q, k, v = (_f64(a) for a in (q, k, v))
    B, n, Hkv, d = k.shape
    Hq = q.shape[1]
    if q.shape != (B, Hq, d) or v.shape != (B, n, Hkv, d):
        raise ValueError("need q [B, Hq, d], k and v [B, n, Hkv, d]")
    if Hq % 2 or Hq % Hkv or (Hq // Hkv) % 2:
        raise ValueError("need Hq even and Hq/Hkv even so each pair shares a KV head")
    lam_logits = _f64(lam_logits)
    if lam_logits.shape != (B, Hq // 2):
        raise ValueError("lam_logits must be [B, Hq/2]")
    lens = np.full(B, n, dtype=np.int64) if lens is None else np.asarray(lens, dtype=np.int64).reshape(-1)
    if lens.shape != (B,) or lens.min(initial=0) < 0 or lens.max(initial=0) > n:
        raise ValueError("lens must be [B] with 0 <= len <= n")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    group = Hq // Hkv
    out = np.zeros((B, Hq // 2, d), dtype=np.float64)
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        for g in range(Hq // 2):
            he, ho = 2 * g, 2 * g + 1
            kv = he // group
            ae = attention_map(q[b, None, he], k[b, :L, kv], scale, False)
            ao = attention_map(q[b, None, ho], k[b, :L, kv], scale, False)
            out[b, g] = ((ae - sigmoid(lam_logits[b, g]) * ao) @ v[b, :L, kv])[0]
    return out


def e4m3_decode(codes) -> np.ndarray:
    """Values of FP8 E4M3 codes ([FP8], the "fn" variant), fp64, same shape.

    Bit 7 is the sign, bits 6..3 the exponent with bias 7, bits 2..0 the
    mantissa.  Exponent 0 is subnormal: (m / 8) * 2^-6.  Otherwise
    (1 + m / 8) * 2^(e - 7), the all-ones exponent included, except that
    exponent 15 with mantissa 7 is NaN (the format has no infinities), so the
    largest finite value is 1.75 * 2^8 = 448.  ``codes``: bytes as a uint8
    array, or a torch uint8 / float8_e4m3fn tensor (its bytes are read).
    """
    x = codes
    if hasattr(x, "detach"):  # a torch tensor: read its bytes
        import torch

        x = x.detach().to("cpu")
        if x.dtype != torch.uint8:
            x = x.view(torch.uint8)
        x = x.numpy()
    c = np.asarray(x)
    if c.dtype != np.uint8:
        raise ValueError("e4m3 codes must be bytes (uint8)")
    c = c.astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def dequant_e4m3(codes, scale: float) -> np.ndarray:
    """A key cache stored as e4m3 codes with one scale per tensor: scale * value ([FP8])."""
    return float(scale) * e4m3_decode(codes)
