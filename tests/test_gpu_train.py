"""GPU parity of the training pair: diffattn_forward_train / diffattn_backward_saved (V1, bf16, d = 64)
and diffattn_v2_forward_train / diffattn_v2_backward_saved (V2, bf16, d = 128).

The training forward must give the forward's output bit for bit (same kernel, extra stores), and
its saved lse must be the base-2 log-sum-exp of the scaled scores (checked against numpy on the
exact bf16 inputs).  The backward from the saved statistics is held to the tensor-core backward's
bar against the fp64 backward oracle: every gradient within 2e-2 max(1, max |ref|) (it differs from
the recomputing backward only by the bf16 rounding of the saved O_1, O_2).
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


def _close(got, ref, name):
    ref = np.asarray(ref, np.float64)
    err = float(np.max(np.abs(got.detach().cpu().double().numpy() - ref)))
    bound = 2e-2 * max(1.0, float(np.max(np.abs(ref))))
    assert err <= bound, f"{name}: max abs error {err} > {bound}"


def _rnd(g, *shape):
    return torch.randn(shape, generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)


def _lse2(q, k, scale, causal):
    """log2 sum_j 2^(scale log2(e) q . k_j) per query row, fp64 (q [n, d], k [n, d])."""
    s = (q.double().cpu().numpy() @ k.double().cpu().numpy().T) * scale * np.log2(np.e)
    if causal:
        s = np.where(np.tril(np.ones_like(s, dtype=bool)), s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    return (m + np.log2(np.exp2(s - m).sum(axis=1, keepdims=True)))[:, 0]


V1 = [  # B, H, n, causal, lambda, gamma
    (1, 1, 1, True, 0.35, True),
    (2, 2, 200, True, 0.35, True),
    (1, 2, 300, False, -0.3, False),
    (1, 1, 1100, True, 1.2, True),
    (2, 4, 257, True, 0.6, True),
]


@pytest.mark.parametrize("B,H,n,causal,lam,gamma", V1)
def test_v1_train_pair(B, H, n, causal, lam, gamma):
    d = 64
    g = torch.Generator(device="cuda").manual_seed(1700 + n + H)
    x = {k: _rnd(g, B, n, H, d) for k in ("q1", "q2", "k1", "k2")}
    x["v"], x["dy"] = _rnd(g, B, n, H, 2 * d), _rnd(g, B, n, H, 2 * d)
    gam = (0.9 + 0.2 * torch.rand(2 * d, generator=g, device="cuda")) if gamma else None
    lam_t = torch.tensor([lam], device="cuda")
    args = (x["q1"], x["q2"], x["k1"], x["k2"], x["v"], lam_t, 0.3)
    out_t, saved = da.diffattn_forward_train(*args, gamma=gam, causal=causal)
    out = da.diffattn_forward(*args, gamma=gam, causal=causal)
    da.device_status()
    assert torch.equal(out_t, out)
    # saved lse of (b, h) rows against numpy
    R = B * H * n
    lse = saved[: 2 * R * 4].view(torch.float32).view(2, B, H, n)
    for b in (0, B - 1):
        for h in (0, H - 1):
            for r_, (qn, kn) in enumerate((("q1", "k1"), ("q2", "k2"))):
                ref = _lse2(x[qn][b, :, h], x[kn][b, :, h], d ** -0.5, causal)
                got = lse[r_, b, h].cpu().double().numpy()
                assert np.max(np.abs(got - ref)) <= 1e-3 * max(1.0, float(np.max(np.abs(ref)))), f"lse_{r_ + 1}"
    got = da.diffattn_backward_saved(*args, x["dy"], saved, gamma=gam, causal=causal)
    da.device_status()
    ref = oracle.diff_attn_v1_backward(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], lam, 0.3,
                                       None if gam is None else gam.cpu(), 1e-5, causal, x["dy"])
    for k in ("dq1", "dq2", "dk1", "dk2", "dv"):
        _close(got[k], ref[k], k)
    _close(got["dlam"][0], ref["dlam"], "dlambda")
    if gamma:
        _close(got["dgamma"], ref["dgamma"], "dgamma")


def test_v1_train_pair_long_items_and_bench_size():
    """n = 9000 (71 query tiles: the forward runs one CTA per item, not the persistent form) bit for bit
    against the forward; B4 H16 n2048 (the bench's backward workload) gradients of two heads against the
    oracle on those heads, dlambda and dgamma against the recomputing backward."""
    g = torch.Generator(device="cuda").manual_seed(1800)
    x = {k: _rnd(g, 1, 9000, 1, 64) for k in ("q1", "q2", "k1", "k2")}
    x["v"] = _rnd(g, 1, 9000, 1, 128)
    lam = torch.tensor([0.3], device="cuda")
    out_t, _ = da.diffattn_forward_train(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], lam, 0.2)
    out = da.diffattn_forward(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], lam, 0.2)
    da.device_status()
    assert torch.equal(out_t, out)

    B, H, n, d = 4, 16, 2048, 64
    x = {k: _rnd(g, B, n, H, d) for k in ("q1", "q2", "k1", "k2")}
    x["v"], x["dy"] = _rnd(g, B, n, H, 2 * d), _rnd(g, B, n, H, 2 * d)
    gam = 0.9 + 0.2 * torch.rand(2 * d, generator=g, device="cuda")
    args = (x["q1"], x["q2"], x["k1"], x["k2"], x["v"], lam, 0.2)
    _, saved = da.diffattn_forward_train(*args, gamma=gam)
    got = da.diffattn_backward_saved(*args, x["dy"], saved, gamma=gam)
    rec = da.diffattn_backward(*args, x["dy"], gamma=gam)
    da.device_status()
    for b in (0, B - 1):
        for h in (0, H - 1):
            sel = {k: t[b:b + 1, :, h:h + 1] for k, t in x.items()}
            ref = oracle.diff_attn_v1_backward(sel["q1"], sel["q2"], sel["k1"], sel["k2"], sel["v"], 0.3, 0.2,
                                               gam.cpu(), 1e-5, True, sel["dy"])
            for k in ("dq1", "dq2", "dk1", "dk2", "dv"):
                _close(got[k][b:b + 1, :, h:h + 1], ref[k], f"{k} b{b} h{h}")
    for k in ("dlam", "dgamma"):
        r_ = rec[k].cpu().double().numpy()
        err = float(np.max(np.abs(got[k].cpu().double().numpy() - r_)))
        assert err <= 2e-2 * max(1.0, float(np.max(np.abs(r_)))), f"{k}: {err}"


V2 = [  # B, Hq, Hkv, n, causal, logit granularity
    (2, 4, 2, 200, True, "token"),
    (1, 8, 2, 300, True, "pair"),
    (2, 4, 2, 129, False, "seq"),
    (1, 4, 2, 1, True, "token"),
]


@pytest.mark.parametrize("B,Hq,Hkv,n,causal,gran", V2)
def test_v2_train_pair(B, Hq, Hkv, n, causal, gran):
    d, G = 128, Hq // 2
    g = torch.Generator(device="cuda").manual_seed(1900 + n + Hq)
    q, k, v, dy = _rnd(g, B, n, Hq, d), _rnd(g, B, n, Hkv, d), _rnd(g, B, n, Hkv, d), _rnd(g, B, n, G, d)
    shape = {"token": (B, n, G), "seq": (B, G), "pair": (G,)}[gran]
    lg = torch.randn(shape, generator=g, device="cuda")
    out_t, saved = da.diffattn_v2_forward_train(q, k, v, lg, causal=causal)
    if gran != "seq":  # diffattn_v2_forward takes [Hq/2] and [B, n, Hq/2] the same way
        out = da.diffattn_v2_forward(q, k, v, lg, causal=causal)
        da.device_status()
        assert torch.equal(out_t, out)
    lg_np = lg.cpu().double().numpy()
    dense = {"token": lambda: lg_np, "seq": lambda: np.broadcast_to(lg_np[:, None, :], (B, n, G)),
             "pair": lambda: np.broadcast_to(lg_np, (B, n, G))}[gran]()
    fwd = oracle.diff_attn_v2(q, k, v, np.ascontiguousarray(dense), causal)
    assert float(np.max(np.abs(out_t.float().cpu().double().numpy() - fwd))) <= 2e-2
    got = da.diffattn_v2_backward_saved(q, k, v, lg, dy, saved, causal=causal)
    da.device_status()
    ref = oracle.diff_attn_v2_backward(q, k, v, np.ascontiguousarray(dense), causal, dy)
    dl = ref["dlogits"]
    if gran == "seq":
        dl = dl.sum(axis=1)
    elif gran == "pair":
        dl = dl.sum(axis=(0, 1))
    for key in ("dq", "dk", "dv"):
        _close(got[key], ref[key], key)
    _close(got["dlogits"], dl, "dlogits")
