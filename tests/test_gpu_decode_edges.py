"""Decode-step edge cases for the warp-wide MMA loop, against the fp64 decode oracles.

The decode kernel keeps a reference maximum per map that moves only when a score exceeds it by
more than 2^8 (log2 domain), and with FP8 key caches it feeds the bf16 query to e4m3 MMAs as two
e4m3 terms after scaling its row by a power of two.  These cases aim at both:
  * scores that climb along the cache (keys aligned with the query, growing with the position), so
    the reference maximum moves many times, for one map while the other stays flat, and with
    ragged lengths that end a climb mid-stage;
  * queries whose elements span many binades, all-zero query rows, and rows of very large and
    very small magnitude (the power-of-two scaling at its clamps).
Bar: 2e-2 max(1, max |ref|) element by element (outputs of nearly one-hot rows are several units
wide; the bf16 rounding of the output alone is half an ulp, 2^-8 |y|).
"""

import numpy as np
import pytest
import torch

import oracle
from differential_attention_03_gb300 import binding as da

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from differential_attention_03_gb300 import build
    build.build()
    torch.cuda.init()


def _np(t):
    return t.detach().float().cpu().double().numpy()


def _check(out, ref, name):
    ref = np.asarray(ref, np.float64)
    err = float(np.max(np.abs(_np(out) - ref)))
    bound = 2e-2 * max(1.0, float(np.max(np.abs(ref))))
    assert np.isfinite(_np(out)).all(), f"{name}: non-finite output"
    assert err <= bound, f"{name}: max abs error {err} > {bound}"


def _quant_e4m3(k):
    """Input preparation: one fp32 scale per tensor (amax / 448) and the e4m3 codes of k / scale."""
    scale = float(k.float().abs().max()) / 448.0
    return (k.float() / scale).to(torch.float8_e4m3fn), scale


def _climbing_keys(g, q, n, slope, noise=0.3):
    """Keys k[b, j, h] = q[b, h] * slope * j / n + noise: the score q . k_j grows along the cache."""
    B, H, d = q.shape
    ramp = torch.linspace(0.0, 1.0, n, device="cuda").view(1, n, 1, 1) * slope
    base = q.float().view(B, 1, H, d) / q.float().norm(dim=-1).clamp_min(1e-6).view(B, 1, H, 1)
    k = base * ramp + noise * torch.randn((B, n, H, d), generator=g, device="cuda")
    return k.to(torch.bfloat16)


@pytest.mark.parametrize("d,n,lens,fp8", [(64, 3000, None, False), (128, 2000, [2000, 1333], False),
                                          (64, 3000, [3000, 77], True), (128, 1500, None, True)])
def test_v1_decode_scores_climbing_along_the_cache(d, n, lens, fp8):
    # Map 1's scores climb by hundreds of log2 units over the cache; map 2's stay flat.
    B, H = 2, 3
    g = torch.Generator(device="cuda").manual_seed(2100 + d + n)
    q1 = torch.randn((B, H, d), generator=g, device="cuda").to(torch.bfloat16)
    q2 = torch.randn((B, H, d), generator=g, device="cuda").to(torch.bfloat16)
    k1 = _climbing_keys(g, q1, n, slope=40.0)
    k2 = torch.randn((B, n, H, d), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((B, n, H, 2 * d), generator=g, device="cuda").to(torch.bfloat16)
    lam = torch.tensor([0.4], device="cuda")
    lens_t = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    if fp8:
        c1, s1 = _quant_e4m3(k1)
        c2, s2 = _quant_e4m3(k2)
        out = da.diffattn_decode_fp8k(q1, q2, c1, c2, s1, s2, v, lam, 0.2, lens=lens_t)
        kk1, kk2 = oracle.dequant_e4m3(c1, s1), oracle.dequant_e4m3(c2, s2)
    else:
        out = da.diffattn_decode(q1, q2, k1, k2, v, lam, 0.2, lens=lens_t)
        kk1, kk2 = k1, k2
    da.device_status()
    ref = oracle.diff_attn_v1_decode(q1, q2, kk1, kk2, v, 0.4, 0.2, None, 1e-5, lens)
    _check(out, ref, f"d{d} fp8={fp8}")


@pytest.mark.parametrize("fp8", [False, True])
def test_v2_decode_scores_climbing_along_the_cache(fp8):
    # The even head of each pair sees climbing scores, the odd head unrelated keys (flat scores).
    B, Hq, Hkv, n, d = 2, 4, 2, 2500, 128
    g = torch.Generator(device="cuda").manual_seed(2200 + int(fp8))
    q = torch.randn((B, Hq, d), generator=g, device="cuda").to(torch.bfloat16)
    qe = q.view(B, Hkv, 2, d)[:, :, 0]
    k = _climbing_keys(g, qe.contiguous(), n, slope=30.0)
    v = torch.randn((B, n, Hkv, d), generator=g, device="cuda").to(torch.bfloat16)
    lg = torch.randn((B, Hq // 2), generator=g, device="cuda")
    if fp8:
        c, s = _quant_e4m3(k)
        out = da.diffattn_v2_decode_fp8k(q, c, s, v, lg)
        kk = oracle.dequant_e4m3(c, s)
    else:
        out = da.diffattn_v2_decode(q, k, v, lg)
        kk = k
    da.device_status()
    ref = oracle.diff_attn_v2_decode(q, kk, v, lg.cpu().double().numpy())
    _check(out, ref, f"v2 fp8={fp8}")


@pytest.mark.parametrize("d", [64, 128])
def test_v1_decode_fp8_keys_query_dynamic_range(d):
    # Query rows: elements spread over 2^-20 .. 2^4 of unit normals; an all-zero row; rows scaled
    # by 1e4 and by 1e-30 (the row scaling's clamps).  The oracle takes the bf16 query as it is.
    B, H, n = 5, 2, 1200
    g = torch.Generator(device="cuda").manual_seed(2300 + d)
    span = torch.exp2(torch.empty((B, H, d), device="cuda").uniform_(-20.0, 4.0, generator=g))
    q1 = torch.randn((B, H, d), generator=g, device="cuda") * span
    q2 = torch.randn((B, H, d), generator=g, device="cuda") * span.flip(-1)
    q1[1] = 0.0
    q1[2] *= 1e4
    q2[3] *= 1e-30
    q1, q2 = q1.to(torch.bfloat16), q2.to(torch.bfloat16)
    k1 = torch.randn((B, n, H, d), generator=g, device="cuda").to(torch.bfloat16)
    k2 = torch.randn((B, n, H, d), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((B, n, H, 2 * d), generator=g, device="cuda").to(torch.bfloat16)
    c1, s1 = _quant_e4m3(k1)
    c2, s2 = _quant_e4m3(k2)
    lam = torch.tensor([0.3], device="cuda")
    out = da.diffattn_decode_fp8k(q1, q2, c1, c2, s1, s2, v, lam, 0.2)
    da.device_status()
    ref = oracle.diff_attn_v1_decode(q1, q2, oracle.dequant_e4m3(c1, s1), oracle.dequant_e4m3(c2, s2), v, 0.3, 0.2,
                                     None, 1e-5, None)
    _check(out, ref, f"d{d}")


def test_v2_decode_fp8_keys_query_dynamic_range():
    B, Hq, Hkv, n, d = 3, 4, 2, 1000, 128
    g = torch.Generator(device="cuda").manual_seed(2400)
    span = torch.exp2(torch.empty((B, Hq, d), device="cuda").uniform_(-20.0, 4.0, generator=g))
    q = torch.randn((B, Hq, d), generator=g, device="cuda") * span
    q[0, 1] = 0.0
    q[1, 2] *= 1e4
    q[2, 3] *= 1e-30
    q = q.to(torch.bfloat16)
    k = torch.randn((B, n, Hkv, d), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((B, n, Hkv, d), generator=g, device="cuda").to(torch.bfloat16)
    c, s = _quant_e4m3(k)
    lg = torch.randn((B, Hq // 2), generator=g, device="cuda")
    out = da.diffattn_v2_decode_fp8k(q, c, s, v, lg)
    da.device_status()
    ref = oracle.diff_attn_v2_decode(q, oracle.dequant_e4m3(c, s), v, lg.cpu().double().numpy())
    _check(out, ref, "v2")
