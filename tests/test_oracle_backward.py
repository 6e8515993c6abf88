"""Pins of the fp64 backward oracle, and planted mistakes that the pins catch.

The backward oracle is the chain rule written out; it is checked against
PyTorch autograd through library routines (scaled_dot_product_attention and
rms_norm, fp64) and against central finite differences of the forward oracle.
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import oracle.backward as ob


def _case(seed, B=2, n=7, H=2, d=4, gamma=True):
    r = np.random.default_rng(seed)
    x = {k: r.normal(size=(B, n, H, d)) for k in ("q1", "q2", "k1", "k2")}
    x["v"] = r.normal(size=(B, n, H, 2 * d))
    x["dy"] = r.normal(size=(B, n, H, 2 * d))
    x["gamma"] = r.uniform(0.5, 1.5, size=2 * d) if gamma else None
    return x


def _autograd(x, lam, lam_init, eps, causal):
    """The forward composed from library routines, differentiated by autograd (fp64)."""
    t = {k: torch.tensor(x[k], dtype=torch.float64, requires_grad=True)
         for k in ("q1", "q2", "k1", "k2", "v")}
    lam_t = torch.tensor(lam, dtype=torch.float64, requires_grad=True)
    d = x["q1"].shape[-1]
    gam = torch.tensor(x["gamma"] if x["gamma"] is not None else np.ones(2 * d), dtype=torch.float64,
                       requires_grad=True)

    def bhsd(a):
        return a.permute(0, 2, 1, 3)
    o1 = F.scaled_dot_product_attention(bhsd(t["q1"]), bhsd(t["k1"]), bhsd(t["v"]), is_causal=causal)
    o2 = F.scaled_dot_product_attention(bhsd(t["q2"]), bhsd(t["k2"]), bhsd(t["v"]), is_causal=causal)
    o = bhsd(o1 - lam_t * o2)
    y = (1.0 - lam_init) * F.rms_norm(o, (2 * d,), weight=gam, eps=eps)
    (y * torch.tensor(x["dy"], dtype=torch.float64)).sum().backward()
    g = {"d" + k: t[k].grad.numpy() for k in t}
    g["dlam"] = float(lam_t.grad)
    g["dgamma"] = gam.grad.numpy()
    return g


CASES = [  # seed, lambda, lambda_init, causal, gamma
    (1, 0.35, 0.2, True, True),
    (2, -0.4, 0.5, True, False),
    (3, 1.3, 0.8, False, True),
    (4, 0.0, 0.2, False, True),
]


@pytest.mark.parametrize("seed,lam,lin,causal,gamma", CASES)
def test_backward_matches_autograd_of_library_routines(seed, lam, lin, causal, gamma):
    x = _case(seed, gamma=gamma)
    got = oracle.diff_attn_v1_backward(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], lam, lin, x["gamma"], 1e-5,
                                       causal, x["dy"])
    want = _autograd(x, lam, lin, 1e-5, causal)
    for k in ("dq1", "dq2", "dk1", "dk2", "dv", "dgamma"):
        np.testing.assert_allclose(got[k], want[k], rtol=1e-9, atol=1e-11, err_msg=k)
    assert got["dlam"] == pytest.approx(want["dlam"], rel=1e-9, abs=1e-11)


def test_backward_matches_finite_differences():
    # Central differences of the forward oracle's loss sum(dy * y), every input element.
    x = _case(7, B=1, n=4, H=1, d=2)
    lam, lin, eps = 0.6, 0.3, 1e-5

    def loss(z, lam_v=lam, gamma=None):
        y = oracle.diff_attn_v1(z["q1"], z["q2"], z["k1"], z["k2"], z["v"], lam_v, lin,
                                x["gamma"] if gamma is None else gamma, eps, True)
        return float(np.sum(y * x["dy"]))
    got = oracle.diff_attn_v1_backward(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], lam, lin, x["gamma"], eps,
                                       True, x["dy"])
    h = 1e-6
    for name in ("q1", "q2", "k1", "k2", "v"):
        fd = np.zeros_like(x[name])
        for idx in np.ndindex(x[name].shape):
            zp = {k: x[k].copy() for k in ("q1", "q2", "k1", "k2", "v")}
            zm = {k: x[k].copy() for k in ("q1", "q2", "k1", "k2", "v")}
            zp[name][idx] += h
            zm[name][idx] -= h
            fd[idx] = (loss(zp) - loss(zm)) / (2 * h)
        np.testing.assert_allclose(got["d" + name], fd, rtol=1e-5, atol=1e-7, err_msg=name)
    base = {k: x[k] for k in ("q1", "q2", "k1", "k2", "v")}
    fd_lam = (loss(base, lam + h) - loss(base, lam - h)) / (2 * h)
    assert got["dlam"] == pytest.approx(fd_lam, rel=1e-5, abs=1e-7)
    fd_g = np.zeros_like(x["gamma"])
    for i in range(fd_g.size):
        gp, gm = x["gamma"].copy(), x["gamma"].copy()
        gp[i] += h
        gm[i] -= h
        fd_g[i] = (loss(base, gamma=gp) - loss(base, gamma=gm)) / (2 * h)
    np.testing.assert_allclose(got["dgamma"], fd_g, rtol=1e-5, atol=1e-7)


def test_lambda_reparam_backward_pins():
    r = np.random.default_rng(9)
    lq1, lk1, lq2, lk2 = (r.normal(0, 0.3, size=6) for _ in range(4))
    got = oracle.lambda_reparam_backward(lq1, lk1, lq2, lk2, 1.7)
    t = [torch.tensor(a, requires_grad=True) for a in (lq1, lk1, lq2, lk2)]
    lam = torch.exp(t[0] @ t[1]) - torch.exp(t[2] @ t[3]) + 0.2
    (1.7 * lam).backward()
    for gi, ti in zip(got, t):
        np.testing.assert_allclose(gi, ti.grad.numpy(), rtol=1e-12)
    # closed form: zero vectors give exp(0) = 1, so d/dlq1 = dlam * lk1
    z = np.zeros(3)
    one = np.array([1.0, 2.0, 3.0])
    g = oracle.lambda_reparam_backward(z, one, z, one, 2.0)
    np.testing.assert_allclose(g[0], 2.0 * one)
    np.testing.assert_allclose(g[2], -2.0 * one)
    np.testing.assert_allclose(g[1], z)


# ------------------------------------------------------------------ planted mistakes
def _mutant(monkeypatch, kind):
    real_map = ob.attention_map

    def run(q1, q2, k1, k2, v, lam, lam_init, gamma, eps, causal, dy):
        q1, q2, k1, k2, v, dy = (ob._f64(a) for a in (q1, q2, k1, k2, v, dy))
        B, n, H, d = q1.shape
        gam = np.ones(2 * d) if gamma is None else ob._f64(gamma)
        m, c = 1.0 - lam_init, 1.0 / math.sqrt(d)
        out = {k: np.zeros_like(q1) for k in ("dq1", "dq2", "dk1", "dk2")}
        out["dv"], dl, dg = np.zeros_like(v), 0.0, np.zeros(2 * d)
        for b in range(B):
            for h in range(H):
                Q1, Q2, K1, K2, V, dY = (t[b, :, h] for t in (q1, q2, k1, k2, v, dy))
                A1, A2 = real_map(Q1, K1, c, causal), real_map(Q2, K2, c, causal)
                O1, O2 = A1 @ V, A2 @ V
                O = O1 - lam * O2
                r = np.sqrt(np.mean(O * O, axis=-1, keepdims=True) + eps)
                Oh, g = O / r, m * gam * dY
                dO = g / r if kind == "norm_no_projection" else (g - Oh * np.mean(g * Oh, -1, keepdims=True)) / r
                dg += np.sum(m * Oh * dY, axis=0)
                out["dv"][b, :, h] = A1.T @ dO - lam * (A2.T @ dO)
                dA1 = dO @ V.T
                dA2 = (dO @ V.T) if kind == "plus_lambda" else -lam * (dO @ V.T)
                dl += -float(np.sum(dO * O2))
                if kind == "no_rowsum":
                    dS1, dS2 = A1 * dA1, A2 * dA2
                else:
                    dS1 = A1 * (dA1 - np.sum(A1 * dA1, -1, keepdims=True))
                    dS2 = A2 * (dA2 - np.sum(A2 * dA2, -1, keepdims=True))
                out["dq1"][b, :, h], out["dq2"][b, :, h] = c * (dS1 @ K1), c * (dS2 @ K2)
                if kind == "transposed_dk":
                    out["dk1"][b, :, h], out["dk2"][b, :, h] = c * (dS1 @ Q1), c * (dS2 @ Q2)
                else:
                    out["dk1"][b, :, h], out["dk2"][b, :, h] = c * (dS1.T @ Q1), c * (dS2.T @ Q2)
        out["dlam"], out["dgamma"] = dl, dg
        return out
    monkeypatch.setattr(oracle, "diff_attn_v1_backward", run)


@pytest.mark.parametrize("kind", ["no_rowsum", "plus_lambda", "transposed_dk", "norm_no_projection"])
def test_backward_pins_catch_mutants(monkeypatch, kind):
    _mutant(monkeypatch, kind)
    with pytest.raises(AssertionError):
        for case in CASES:
            test_backward_matches_autograd_of_library_routines(*case)


def test_mutant_harness_is_faithful(monkeypatch):
    # The harness without a planted mistake passes the pin (so a failure above is the mistake's).
    _mutant(monkeypatch, "none")
    for case in CASES:
        test_backward_matches_autograd_of_library_routines(*case)


# ------------------------------------------------------------------ DIFF V2
def _v2_autograd(x, causal):
    """V2 composed from library routines (SDPA per query head over its KV head), autograd in fp64."""
    q = torch.tensor(x["q"], requires_grad=True)
    k = torch.tensor(x["k"], requires_grad=True)
    v = torch.tensor(x["v"], requires_grad=True)
    lg = torch.tensor(x["lg"], requires_grad=True)
    B, n, Hq, d = q.shape
    group = Hq // k.shape[2]
    kk = k.repeat_interleave(group, dim=2)  # query head j reads KV head j // group
    vv = v.repeat_interleave(group, dim=2)
    a = F.scaled_dot_product_attention(q.permute(0, 2, 1, 3), kk.permute(0, 2, 1, 3), vv.permute(0, 2, 1, 3),
                                       is_causal=causal).permute(0, 2, 1, 3)
    y = a[:, :, 0::2] - torch.sigmoid(lg)[..., None] * a[:, :, 1::2]
    (y * torch.tensor(x["dy"])).sum().backward()
    return {"dq": q.grad.numpy(), "dk": k.grad.numpy(), "dv": v.grad.numpy(), "dlogits": lg.grad.numpy()}


def _v2_case(seed, B=2, n=6, Hq=4, Hkv=2, d=4):
    r = np.random.default_rng(seed)
    return {"q": r.normal(size=(B, n, Hq, d)), "k": r.normal(size=(B, n, Hkv, d)), "v": r.normal(size=(B, n, Hkv, d)),
            "lg": r.normal(size=(B, n, Hq // 2)), "dy": r.normal(size=(B, n, Hq // 2, d))}


@pytest.mark.parametrize("Hq,Hkv,causal", [(4, 2, True), (8, 2, True), (4, 1, False), (2, 1, True)])
def test_v2_backward_matches_autograd(Hq, Hkv, causal):
    x = _v2_case(20 + Hq + Hkv, Hq=Hq, Hkv=Hkv)
    got = oracle.diff_attn_v2_backward(x["q"], x["k"], x["v"], x["lg"], causal, x["dy"])
    want = _v2_autograd(x, causal)
    for key in ("dq", "dk", "dv", "dlogits"):
        np.testing.assert_allclose(got[key], want[key], rtol=1e-9, atol=1e-11, err_msg=key)


def test_v2_backward_matches_finite_differences():
    x = _v2_case(31, B=1, n=4, Hq=4, Hkv=1, d=2)
    got = oracle.diff_attn_v2_backward(x["q"], x["k"], x["v"], x["lg"], True, x["dy"])

    def loss(z):
        return float(np.sum(oracle.diff_attn_v2(z["q"], z["k"], z["v"], z["lg"], True) * x["dy"]))
    h = 1e-6
    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("lg", "dlogits")):
        fd = np.zeros_like(x[name])
        for idx in np.ndindex(x[name].shape):
            zp = {kk: x[kk].copy() for kk in ("q", "k", "v", "lg")}
            zm = {kk: x[kk].copy() for kk in ("q", "k", "v", "lg")}
            zp[name][idx] += h
            zm[name][idx] -= h
            fd[idx] = (loss(zp) - loss(zm)) / (2 * h)
        np.testing.assert_allclose(got[gname], fd, rtol=1e-5, atol=1e-7, err_msg=name)


def test_v2_backward_pin_catches_unsummed_kv_gradient(monkeypatch):
    # A plausible mistake: dK / dV of a KV head taken from its last pair only (not summed over the group).
    real = ob.diff_attn_v2_backward

    def last_pair_only(q, k, v, lam_logits, causal, dy, scale=None):
        out = real(q, k, v, lam_logits, causal, dy, scale)
        G, Hkv = np.asarray(lam_logits).shape[2], np.asarray(k).shape[2]
        if G > Hkv:  # several pairs per KV head: keep one pair's share
            q1 = np.asarray(q).copy()
            q1[:, :, :-2] = 0.0
            one = real(q1, k, v, lam_logits, causal, dy, scale)
            out["dk"] = one["dk"]
        return out
    monkeypatch.setattr(oracle, "diff_attn_v2_backward", last_pair_only)
    with pytest.raises(AssertionError):
        test_v2_backward_matches_autograd(8, 2, True)
