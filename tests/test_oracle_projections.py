"""Pins of the attention-layer oracle (projections in, W^O out).

Against the layer composed from PyTorch library routines in fp64 (linear,
scaled_dot_product_attention, rms_norm), and against an invariant that a
head-indexing mistake breaks: permuting the heads consistently in W^Q, W^K,
W^V and W^O leaves the layer's output unchanged.
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import oracle.projections as op


def _v1_weights(seed, D=12, H=3, d=4):
    r = np.random.default_rng(seed)
    w = {k: r.normal(0, 0.4, size=(D, H * 2 * d)) for k in ("wq", "wk", "wv")}
    w["wo"] = r.normal(0, 0.4, size=(H * 2 * d, D))
    for k in ("lq1", "lk1", "lq2", "lk2"):
        w[k] = r.normal(0, 0.1, size=d)
    w["gamma"] = r.uniform(0.8, 1.2, size=2 * d)
    return w


def _torch_v1(x, w, lam_init, H, causal):
    t = {k: torch.tensor(v) for k, v in w.items()}
    xt = torch.tensor(x)
    B, n, D = x.shape
    d = w["wq"].shape[1] // (2 * H)
    q = F.linear(xt, t["wq"].T).view(B, n, H, 2 * d).transpose(1, 2)
    k = F.linear(xt, t["wk"].T).view(B, n, H, 2 * d).transpose(1, 2)
    v = F.linear(xt, t["wv"].T).view(B, n, H, 2 * d).transpose(1, 2)
    lam = torch.exp(t["lq1"] @ t["lk1"]) - torch.exp(t["lq2"] @ t["lk2"]) + lam_init
    a1 = F.scaled_dot_product_attention(q[..., :d], k[..., :d], v, is_causal=causal)
    a2 = F.scaled_dot_product_attention(q[..., d:], k[..., d:], v, is_causal=causal)
    o = (a1 - lam * a2).transpose(1, 2)  # [B, n, H, 2d]
    y = (1 - lam_init) * F.rms_norm(o, (2 * d,), weight=t["gamma"], eps=1e-5)
    return F.linear(y.reshape(B, n, H * 2 * d), t["wo"].T).numpy()


@pytest.mark.parametrize("causal", [True, False])
def test_v1_layer_matches_library_composition(causal):
    w = _v1_weights(3)
    x = np.random.default_rng(4).normal(size=(2, 7, 12))
    got = oracle.diff_v1_layer(x, w["wq"], w["wk"], w["wv"], w["wo"], w["lq1"], w["lk1"], w["lq2"], w["lk2"], 0.35,
                               3, w["gamma"], 1e-5, causal)
    np.testing.assert_allclose(got, _torch_v1(x, w, 0.35, 3, causal), rtol=1e-10, atol=1e-12)


def test_v1_layer_head_permutation_invariance():
    w = _v1_weights(5)
    x = np.random.default_rng(6).normal(size=(1, 6, 12))
    H, d = 3, 4
    perm = [2, 0, 1]
    cols = np.concatenate([np.arange(h * 2 * d, (h + 1) * 2 * d) for h in perm])
    args = (w["lq1"], w["lk1"], w["lq2"], w["lk2"], 0.5, H, w["gamma"])
    a = oracle.diff_v1_layer(x, w["wq"], w["wk"], w["wv"], w["wo"], *args)
    b = oracle.diff_v1_layer(x, w["wq"][:, cols], w["wk"][:, cols], w["wv"][:, cols], w["wo"][cols], *args)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)
    # Permuting W^O alone must change the output (the pin sees the head order).
    c = oracle.diff_v1_layer(x, w["wq"], w["wk"], w["wv"], w["wo"][cols], *args)
    assert np.max(np.abs(a - c)) > 1e-3


def _v2_weights(seed, D=10, Hq=4, Hkv=2, d=4):
    r = np.random.default_rng(seed)
    return {"wq": r.normal(0, 0.4, size=(D, Hq * d)), "wk": r.normal(0, 0.4, size=(D, Hkv * d)),
            "wv": r.normal(0, 0.4, size=(D, Hkv * d)), "wl": r.normal(0, 0.4, size=(D, Hq // 2)),
            "wo": r.normal(0, 0.4, size=(Hq // 2 * d, D))}


@pytest.mark.parametrize("Hq,Hkv,causal", [(4, 2, True), (8, 2, True), (4, 1, False)])
def test_v2_layer_matches_library_composition(Hq, Hkv, causal):
    w = _v2_weights(7 + Hq, Hq=Hq, Hkv=Hkv)
    x = np.random.default_rng(8).normal(size=(2, 6, 10))
    got = oracle.diff_v2_layer(x, w["wq"], w["wk"], w["wv"], w["wl"], w["wo"], Hq, Hkv, causal)
    t = {k: torch.tensor(v) for k, v in w.items()}
    xt = torch.tensor(x)
    B, n, D = x.shape
    d = w["wq"].shape[1] // Hq
    q = F.linear(xt, t["wq"].T).view(B, n, Hq, d).transpose(1, 2)
    k = F.linear(xt, t["wk"].T).view(B, n, Hkv, d).transpose(1, 2).repeat_interleave(Hq // Hkv, dim=1)
    v = F.linear(xt, t["wv"].T).view(B, n, Hkv, d).transpose(1, 2).repeat_interleave(Hq // Hkv, dim=1)
    a = F.scaled_dot_product_attention(q, k, v, is_causal=causal).transpose(1, 2)  # [B, n, Hq, d]
    s = torch.sigmoid(F.linear(xt, t["wl"].T))[..., None]  # [B, n, Hq/2, 1]
    y = a[:, :, 0::2] - s * a[:, :, 1::2]
    want = F.linear(y.reshape(B, n, Hq // 2 * d), t["wo"].T).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)


def test_layers_check_shapes():
    w = _v1_weights(1)
    with pytest.raises(ValueError):
        oracle.diff_v1_layer(np.zeros((1, 2, 11)), w["wq"], w["wk"], w["wv"], w["wo"], w["lq1"], w["lk1"],
                             w["lq2"], w["lk2"], 0.2, 3)
    assert math.isfinite(float(oracle.diff_v1_layer(np.ones((1, 2, 12)), w["wq"], w["wk"], w["wv"], w["wo"],
                                                    w["lq1"], w["lk1"], w["lq2"], w["lk2"], 0.2, 3).sum()))


def test_v1_layer_pin_catches_swapped_halves(monkeypatch):
    # A plausible mistake: Q_1 taken from the second half of the head's projection.
    real = op.diff_attn_v1

    def swapped(q1, q2, k1, k2, v, lam, lam_init, gamma=None, eps=1e-5, causal=True, rows=None):
        return real(q2, q1, k1, k2, v, lam, lam_init, gamma, eps, causal, rows)
    monkeypatch.setattr(op, "diff_attn_v1", swapped)
    with pytest.raises(AssertionError):
        test_v1_layer_matches_library_composition(True)
