"""Pins of the fp64 CPU oracle to what the pages and the mathematics fix.

None of these tests re-types the oracle's formulas: each compares it with a
value the pages print, a closed form, an invariant, a library routine
(torch SDPA / rms_norm in fp64) or brute-force scalar loops.
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _worked_example_inputs():
    fx = json.load(open(os.path.join(GOLDEN, "worked_example.json")))
    torch.manual_seed(0)
    n, d = fx["n"], fx["d"]
    q1, k1, q2, k2 = torch.randn(4, n, d)
    v = torch.randn(n, 2 * d)
    return fx, q1, k1, q2, k2, v


# ---------------------------------------------------------------- worked example
def test_worked_example_printed_result():
    """Glossary page, 'How differential attention works': row sum 0.20, 13 of 36 negative."""
    fx, q1, k1, q2, k2, v = _worked_example_inputs()
    dmap = oracle.difference_map(q1, k1, q2, k2, fx["lambda"], causal=fx["causal"])
    assert dmap.shape == (fx["n"], fx["n"])
    assert f"{dmap.sum(axis=-1)[0]:.2f}" == fx["row_sum_2dp"]
    assert int((dmap < 0).sum()) == fx["negative_weights"]
    assert dmap.size == fx["total_weights"]
    # Every row (not only the printed first one) sums to 1 - lambda.
    np.testing.assert_allclose(dmap.sum(axis=-1), 1 - fx["lambda"], atol=1e-12)


def test_worked_example_rejects_other_scales():
    """A planted mistake in the scale (none, or 1/sqrt(2d)) changes the printed count."""
    fx, q1, k1, q2, k2, v = _worked_example_inputs()
    for wrong in (1.0, 1.0 / math.sqrt(2 * fx["d"])):
        dmap = oracle.difference_map(q1, k1, q2, k2, fx["lambda"], causal=False, scale=wrong)
        assert int((dmap < 0).sum()) != fx["negative_weights"]


# ---------------------------------------------------------------- lambda
def test_lambda_init_properties():
    """lambda_init starts at 0.2 (l = 1), rises toward 0.8 with depth, stays in (0, 1)."""
    assert oracle.lambda_init(1) == pytest.approx(0.2, abs=1e-15)
    vals = [oracle.lambda_init(l) for l in range(1, 100)]
    assert all(0.0 < x < 0.8 for x in vals)
    assert all(b > a for a, b in zip(vals, vals[1:]))
    assert oracle.lambda_init(200) == pytest.approx(0.8, abs=1e-12)
    # The gap to 0.8 shrinks by the same factor every layer (an exponential in l).
    gaps = [0.8 - x for x in vals[:30]]
    ratios = [b / a for a, b in zip(gaps, gaps[1:])]
    assert max(ratios) - min(ratios) < 1e-12
    with pytest.raises(ValueError):
        oracle.lambda_init(0)


# lambda_init at the layers of the measured workloads, evaluated from the schedule
# the news article prints (section "差分注意力": 0.8 - 0.6 exp(-0.3 (l - 1)),
# l in [1, L]) and the glossary's prose after its worked example (the same
# schedule, deeper layers starting nearer 0.8).  Written out as literals so that
# a wrong rate or a wrong layer offset in the oracle cannot reproduce them.
LAMBDA_INIT_CLOSED_FORMS = {
    1: 0.2,
    4: 0.5560582041556406,    # 0.8 - 0.6 e^-0.9
    12: 0.777870099559256,    # 0.8 - 0.6 e^-3.3
    20: 0.7979924207255172,   # 0.8 - 0.6 e^-5.7
}
# The gap 0.8 - lambda_init shrinks by e^-0.3 per layer.
LAMBDA_INIT_GAP_RATIO = 0.7408182206817179


def test_lambda_init_closed_forms():
    """The rate 0.3 and the offset (l - 1) of the schedule, pinned by its values at l = 1, 4, 12, 20."""
    for l, want in LAMBDA_INIT_CLOSED_FORMS.items():
        assert abs(oracle.lambda_init(l) - want) <= 1e-15, l
    g1, g2 = 0.8 - oracle.lambda_init(7), 0.8 - oracle.lambda_init(8)
    assert abs(g2 / g1 - LAMBDA_INIT_GAP_RATIO) <= 1e-13


def test_lambda_reparam_closed_forms():
    lin = 0.5560582041556406
    z = np.zeros(64)
    assert oracle.lambda_reparam(z, z, z, z, lin) == pytest.approx(lin, abs=1e-15)
    # exp(ln 2) - exp(0) + lambda_init = 1 + lambda_init
    a = np.zeros(8)
    a[3] = math.sqrt(math.log(2.0))
    assert oracle.lambda_reparam(a, a, np.zeros(8), np.zeros(8), lin) == pytest.approx(1 + lin, abs=1e-14)
    # Swapping the two pairs mirrors lambda about lambda_init.
    r = _rng(1)
    v = [r.normal(0, 0.1, 64) for _ in range(4)]
    lam = oracle.lambda_reparam(*v, lin)
    lam_sw = oracle.lambda_reparam(v[2], v[3], v[0], v[1], lin)
    assert lam + lam_sw == pytest.approx(2 * lin, abs=1e-14)
    # Equal inner products cancel; the pairing is q1 with k1 (not q1 with q2).
    assert oracle.lambda_reparam(v[0], v[1], v[1], v[0], lin) == pytest.approx(lin, abs=1e-15)
    lam_x = oracle.lambda_reparam(v[0], v[2], v[1], v[3], lin)
    assert abs(lam_x - lam) > 1e-6


# ---------------------------------------------------------------- difference map
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("lam", [0.8, -0.3, 1.7])
def test_rows_sum_to_one_minus_lambda(causal, lam):
    """Glossary page: each map sums to 1, so each row of the difference sums to 1 - lambda."""
    r = _rng(2)
    n, d = 37, 16
    q1, k1, q2, k2 = (r.normal(size=(n, d)) for _ in range(4))
    dmap = oracle.difference_map(q1, k1, q2, k2, lam, causal)
    np.testing.assert_allclose(dmap.sum(-1), 1 - lam, atol=1e-12)
    if causal:
        assert np.all(np.triu(dmap, 1) == 0)


@pytest.mark.parametrize("causal", [False, True])
def test_lambda_zero_is_sdpa(causal):
    """lambda = 0 leaves one ordinary softmax attention (torch SDPA, fp64, V width 2d)."""
    r = _rng(3)
    n, d = 150, 32  # 150 > the oracle's 128-row block: exercises two blocks
    q1, q2, k1, k2 = (r.normal(size=(n, d)) for _ in range(4))
    v = r.normal(size=(n, 2 * d))
    o = oracle.diff_attn_head(q1, q2, k1, k2, v, 0.0, causal)
    t = lambda a: torch.from_numpy(a)[None, None]
    ref = F.scaled_dot_product_attention(t(q1), t(k1), t(v), is_causal=causal)[0, 0].numpy()
    np.testing.assert_allclose(o, ref, atol=1e-12, rtol=0)


def test_equal_maps_reduce_to_scaled_attention():
    """Q1 = Q2 and K1 = K2 give D = (1 - lambda) A and a sign-flipped norm when lambda > 1."""
    r = _rng(4)
    B, n, H, d = 1, 40, 2, 8
    q = r.normal(size=(B, n, H, d))
    k = r.normal(size=(B, n, H, d))
    v = r.normal(size=(B, n, H, 2 * d))
    for lam in (0.3, 1.4):
        y = oracle.diff_attn_v1(q, q, k, k, v, lam, 0.2, causal=True, eps=0.0)
        for h in range(H):
            t = lambda a: torch.from_numpy(np.ascontiguousarray(a[0, :, h]))[None, None]
            att = F.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True)[0, 0]
            ref = F.rms_norm(att, (2 * d,), eps=0.0).numpy() * math.copysign(1, 1 - lam) * 0.8
            np.testing.assert_allclose(y[0, :, h], ref, atol=1e-12)


def test_causal_row_zero_closed_form():
    """Row 0 sees only key 0: y0 = (1-lambda_init) g (1-lambda) v0 / sqrt((1-lambda)^2 ms(v0) + eps)."""
    r = _rng(5)
    B, n, H, d = 2, 9, 3, 4
    q1, q2, k1, k2 = (r.normal(size=(B, n, H, d)) for _ in range(4))
    v = r.normal(size=(B, n, H, 2 * d))
    gamma = r.uniform(0.9, 1.1, 2 * d)
    lam, lin, eps = 0.37, 0.77787, 1e-5
    y = oracle.diff_attn_v1(q1, q2, k1, k2, v, lam, lin, gamma, eps, causal=True, rows=[0])
    for b in range(B):
        for h in range(H):
            v0 = v[b, 0, h]
            want = (1 - lin) * gamma * (1 - lam) * v0 / math.sqrt((1 - lam) ** 2 * np.mean(v0 ** 2) + eps)
            np.testing.assert_allclose(y[b, 0, h], want, atol=1e-13)


def test_zero_queries_give_running_means():
    """Q = 0 makes both maps uniform over the visible keys: O_i = (1-lambda) mean_{j<=i} v_j."""
    r = _rng(6)
    n, d = 20, 4
    z = np.zeros((n, d))
    k1, k2 = r.normal(size=(n, d)), r.normal(size=(n, d))
    v = r.normal(size=(n, 2 * d))
    lam = 0.6
    o = oracle.diff_attn_head(z, z, k1, k2, v, lam, causal=True)
    want = (1 - lam) * np.cumsum(v, axis=0) / np.arange(1, n + 1)[:, None]
    np.testing.assert_allclose(o, want, atol=1e-13)
    o_nc = oracle.diff_attn_head(z, z, k1, k2, v, lam, causal=False)
    np.testing.assert_allclose(o_nc, np.broadcast_to((1 - lam) * v.mean(0), o_nc.shape), atol=1e-13)


def test_softmax_row_norm_bounds():
    """V2 page, context-RMS table: a softmax row's 2-norm lies in [1/sqrt(visible), 1]."""
    r = _rng(7)
    n, d = 300, 16
    q, k = r.normal(size=(n, d)) * 2, r.normal(size=(n, d)) * 2
    a = oracle.attention_map(q, k, 1 / 4, causal=True)
    norms = np.linalg.norm(a, axis=-1)
    lo = 1 / np.sqrt(np.arange(1, n + 1))
    assert np.all(norms >= lo - 1e-12) and np.all(norms <= 1 + 1e-12)
    np.testing.assert_allclose(a.sum(-1), 1, atol=1e-12)
    assert np.all(a >= 0)


# ---------------------------------------------------------------- RMSNorm
def test_head_rmsnorm_matches_torch_rms_norm():
    r = _rng(8)
    o = r.normal(size=(33, 256)) * 0.05
    gamma = r.uniform(0.9, 1.1, 256)
    lin, eps = 0.7979924207255172, 1e-5
    y = oracle.head_rmsnorm(o, gamma, eps, lin)
    ref = F.rms_norm(torch.from_numpy(o), (256,), torch.from_numpy(gamma), eps).numpy() * (1 - lin)
    np.testing.assert_allclose(y, ref, atol=1e-13)
    # Mean square with gamma = 1: (1-lambda_init)^2 m / (m + eps).
    y1 = oracle.head_rmsnorm(o, None, eps, lin)
    m = np.mean(o ** 2, -1)
    np.testing.assert_allclose(np.mean(y1 ** 2, -1), (1 - lin) ** 2 * m / (m + eps), rtol=1e-12)


def test_v1_norm_is_per_head_and_per_token():
    """Scaling one head's V by c leaves that head's normalised output (eps = 0) and others unchanged."""
    r = _rng(9)
    B, n, H, d = 1, 12, 3, 4
    q1, q2, k1, k2 = (r.normal(size=(B, n, H, d)) for _ in range(4))
    v = r.normal(size=(B, n, H, 2 * d))
    y = oracle.diff_attn_v1(q1, q2, k1, k2, v, 0.5, 0.2, eps=0.0)
    v2 = v.copy()
    v2[:, :, 1] *= 7.0
    y2 = oracle.diff_attn_v1(q1, q2, k1, k2, v2, 0.5, 0.2, eps=0.0)
    np.testing.assert_allclose(y2, y, atol=1e-12)


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("causal", [True, False])
def test_v1_matches_brute_force(causal):
    r = _rng(10)
    B, n, H, d = 2, 7, 2, 4
    q1, q2, k1, k2 = (r.normal(size=(B, n, H, d)) for _ in range(4))
    v = r.normal(size=(B, n, H, 2 * d))
    gamma = r.uniform(0.9, 1.1, 2 * d)
    lam, lin = 0.65, 0.5560582041556406
    y = oracle.diff_attn_v1(q1, q2, k1, k2, v, lam, lin, gamma, 1e-5, causal)
    yb = np.array(brute.brute_v1(q1, q2, k1, k2, v, lam, lin, gamma, 1e-5, causal))
    np.testing.assert_allclose(y, yb, atol=1e-12)
    rows = [6, 0, 3]
    np.testing.assert_allclose(
        oracle.diff_attn_v1(q1, q2, k1, k2, v, lam, lin, gamma, 1e-5, causal, rows=rows), yb[:, rows], atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("hq,hkv", [(4, 2), (8, 2), (4, 1)])
def test_v2_matches_brute_force(causal, hq, hkv):
    r = _rng(11)
    B, n, d = 2, 6, 4
    q = r.normal(size=(B, n, hq, d))
    k = r.normal(size=(B, n, hkv, d))
    v = r.normal(size=(B, n, hkv, d))
    logits = r.normal(size=(B, n, hq // 2))
    out = oracle.diff_attn_v2(q, k, v, logits, causal)
    ob = np.array(brute.brute_v2(q, k, v, logits, causal))
    np.testing.assert_allclose(out, ob, atol=1e-12)


# ---------------------------------------------------------------- DIFF V2
def _gqa_sdpa(q, k, v, causal):
    """torch SDPA (fp64) with KV heads repeated for grouped-query attention."""
    g = q.shape[2] // k.shape[2]
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).transpose(1, 2)
    kk = t(k).repeat_interleave(g, dim=1)
    vv = t(v).repeat_interleave(g, dim=1)
    return F.scaled_dot_product_attention(t(q), kk, vv, is_causal=causal).transpose(1, 2).numpy()


@pytest.mark.parametrize("causal", [True, False])
def test_v2_against_sdpa(causal):
    """out_g = SDPA head 2g - sigmoid(logit) * SDPA head 2g+1; a very negative logit leaves head 2g."""
    r = _rng(12)
    B, n, hq, hkv, d = 2, 140, 8, 2, 16
    q = r.normal(size=(B, n, hq, d))
    k = r.normal(size=(B, n, hkv, d))
    v = r.normal(size=(B, n, hkv, d))
    att = _gqa_sdpa(q, k, v, causal)
    logits = r.normal(size=(B, n, hq // 2))
    out = oracle.diff_attn_v2(q, k, v, logits, causal)
    sig = 1 / (1 + np.exp(-logits))
    np.testing.assert_allclose(out, att[:, :, 0::2] - sig[..., None] * att[:, :, 1::2], atol=1e-12)
    off = oracle.diff_attn_v2(q, k, v, np.full((B, n, hq // 2), -60.0), causal)
    np.testing.assert_allclose(off, att[:, :, 0::2], atol=1e-12)


def test_v2_wrong_pairing_differs():
    """The first-half/second-half split mixes KV groups and gives a different output."""
    r = _rng(13)
    B, n, hq, hkv, d = 1, 30, 8, 4, 8
    q = r.normal(size=(B, n, hq, d))
    k = r.normal(size=(B, n, hkv, d))
    v = r.normal(size=(B, n, hkv, d))
    logits = r.normal(size=(B, n, hq // 2))
    good = oracle.diff_attn_v2(q, k, v, logits)
    bad = oracle.diff_attn_v2(q, k, v, logits, pairing="halves")
    assert np.max(np.abs(good - bad)) > 0.1


def test_v2_difference_rows_below_sqrt2():
    """V2 page, context-RMS table: ||A_even - sigmoid * A_odd||_2 < sqrt(2)."""
    r = _rng(14)
    n, d = 200, 8
    q1, q2, k = (r.normal(size=(n, d)) * 3 for _ in range(3))
    for logit in (-3.0, 0.0, 5.0):
        s = 1 / (1 + math.exp(-logit))
        dm = oracle.attention_map(q1, k, 1 / math.sqrt(d), True) - s * oracle.attention_map(q2, k, 1 / math.sqrt(d), True)
        norms = np.linalg.norm(dm, axis=-1)
        assert np.all(norms < math.sqrt(2)) and np.all(norms >= 0)


def test_v2_rejects_pairs_that_straddle_groups():
    q = np.zeros((1, 4, 6, 2))
    k = np.zeros((1, 4, 2, 2))
    with pytest.raises(ValueError):
        oracle.diff_attn_v2(q, k, k, np.zeros((1, 4, 3)))


# ---------------------------------------------------------------- decode (one query per sequence)
def _decode_case(seed, B=3, n=9, H=2, d=4):
    r = _rng(seed)
    q1, q2 = (r.normal(size=(B, H, d)) for _ in range(2))
    k1, k2 = (r.normal(size=(B, n, H, d)) for _ in range(2))
    v = r.normal(size=(B, n, H, 2 * d))
    return q1, q2, k1, k2, v, r.uniform(0.9, 1.1, 2 * d)


def test_decode_is_the_last_row_of_causal_attention():
    # The new token's query over the cache (its own key included) is the last
    # row of the causal forward over the sequence with that query appended.
    q1, q2, k1, k2, v, g = _decode_case(30)
    B, n, H, d = k1.shape
    r = _rng(31)
    Q1, Q2 = (r.normal(size=(B, n, H, d)) for _ in range(2))
    Q1[:, -1], Q2[:, -1] = q1, q2
    lam, lin = 0.41, 0.2
    full = oracle.diff_attn_v1(Q1, Q2, k1, k2, v, lam, lin, g, 1e-5, True, rows=[n - 1])[:, 0]
    np.testing.assert_allclose(oracle.diff_attn_v1_decode(q1, q2, k1, k2, v, lam, lin, g), full, atol=1e-12)


def test_decode_matches_brute_force_with_lengths():
    q1, q2, k1, k2, v, g = _decode_case(32)
    lens = [9, 1, 5]
    lam, lin = 0.7, 0.5560582041556406
    y = oracle.diff_attn_v1_decode(q1, q2, k1, k2, v, lam, lin, g, 1e-5, lens)
    yb = np.array(brute.brute_v1_decode(q1, q2, k1, k2, v, lam, lin, g, 1e-5, lens))
    np.testing.assert_allclose(y, yb, atol=1e-12)


def test_decode_closed_forms():
    q1, q2, k1, k2, v, _ = _decode_case(33)
    B, n, H, d = k1.shape
    lam, lin, eps = 0.3, 0.2, 1e-5
    # Zero queries: both maps are uniform over the visible keys, O = (1 - lambda) mean(V).
    z = np.zeros_like(q1)
    lens = np.array([9, 4, 1])
    y = oracle.diff_attn_v1_decode(z, z, k1, k2, v, lam, lin, None, eps, lens)
    for b in range(B):
        o = (1 - lam) * v[b, :lens[b]].mean(axis=0)  # [H, 2d]
        want = (1 - lin) * o / np.sqrt((o * o).mean(axis=-1, keepdims=True) + eps)
        np.testing.assert_allclose(y[b], want, atol=1e-12)
    # One visible key: both maps put weight 1 on it, O = (1 - lambda) V[0].
    y1 = oracle.diff_attn_v1_decode(q1, q2, k1, k2, v, lam, lin, None, eps, [1, 1, 1])
    o = (1 - lam) * v[:, 0]
    np.testing.assert_allclose(y1, (1 - lin) * o / np.sqrt((o * o).mean(axis=-1, keepdims=True) + eps), atol=1e-12)
    # No visible key: zeros (the reading for an empty cache).
    assert not np.any(oracle.diff_attn_v1_decode(q1, q2, k1, k2, v, lam, lin, None, eps, [0, 9, 0])[[0, 2]])


def test_v2_decode_is_the_last_row_of_causal_v2():
    r = _rng(40)
    B, n, Hq, Hkv, d = 2, 7, 8, 2, 4
    Q = r.normal(size=(B, n, Hq, d))
    k, v = r.normal(size=(B, n, Hkv, d)), r.normal(size=(B, n, Hkv, d))
    lg = r.normal(size=(B, n, Hq // 2))
    full = oracle.diff_attn_v2(Q, k, v, lg, True, rows=[n - 1])[:, 0]
    y = oracle.diff_attn_v2_decode(Q[:, -1], k, v, lg[:, -1])
    np.testing.assert_allclose(y, full, atol=1e-12)


def test_v2_decode_lengths_and_closed_forms():
    r = _rng(41)
    B, n, Hq, Hkv, d = 3, 6, 4, 1, 4
    q = r.normal(size=(B, Hq, d))
    k, v = r.normal(size=(B, n, Hkv, d)), r.normal(size=(B, n, Hkv, d))
    lg = r.normal(size=(B, Hq // 2))
    lens = [6, 2, 0]
    y = oracle.diff_attn_v2_decode(q, k, v, lg, lens)
    # Against the full-sequence oracle on the truncated cache, row by row.
    for b, L in enumerate(lens):
        if L == 0:
            assert not np.any(y[b])
            continue
        Q = np.zeros((1, L, Hq, d))
        Q[0, -1] = q[b]
        lgs = np.zeros((1, L, Hq // 2))
        lgs[0, -1] = lg[b]
        np.testing.assert_allclose(y[b], oracle.diff_attn_v2(Q, k[b:b + 1, :L], v[b:b + 1, :L], lgs, True,
                                                             rows=[L - 1])[0, 0], atol=1e-12)
    # Zero queries: uniform maps, out = (1 - sigmoid(logit)) mean(V) of the pair's KV head.
    z = oracle.diff_attn_v2_decode(np.zeros_like(q), k, v, lg, [6, 3, 1])
    for b, L in enumerate([6, 3, 1]):
        for g in range(Hq // 2):
            want = (1 - 1 / (1 + math.exp(-lg[b, g]))) * v[b, :L, 0].mean(axis=0)
            np.testing.assert_allclose(z[b, g], want, atol=1e-12)


# ---------------------------------------------------------------- FP8 (e4m3) key-cache codes
def test_e4m3_decode_closed_forms():
    # Values the E4M3 format fixes: zero and negative zero, one, the largest
    # finite value, the smallest normal and subnormal values, NaN, sign symmetry.
    v = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert v[0x00] == 0.0 and v[0x80] == 0.0 and math.copysign(1.0, v[0x80]) == -1.0
    assert v[0x38] == 1.0 and v[0xB8] == -1.0
    assert v[0x30] == 0.5 and v[0x40] == 2.0 and v[0x3C] == 1.5
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert v[0x08] == 2.0 ** -6 and v[0x01] == 2.0 ** -9 and v[0x07] == 7 * 2.0 ** -9
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF]) and np.isnan(v).sum() == 2
    np.testing.assert_array_equal(v[0x80:0xFF], -v[0x00:0x7F])
    assert np.all(np.diff(v[0x00:0x7F]) > 0)  # finite positive codes increase with the code


def test_e4m3_decode_matches_torch_float8():
    # Every code against PyTorch's own float8_e4m3fn conversion (a library routine).
    c = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    want = c.view(torch.float8_e4m3fn).double().numpy()
    got = oracle.e4m3_decode(c.numpy())
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(got[ok], want[ok])
    # A float8 tensor is read through its bytes; dequantisation multiplies by the scale.
    x = torch.tensor([[0.75, -3.5], [448.0, 2.0 ** -9]]).to(torch.float8_e4m3fn)
    np.testing.assert_array_equal(oracle.dequant_e4m3(x, 0.25), 0.25 * np.array([[0.75, -3.5], [448.0, 2.0 ** -9]]))
