"""GPU parity of the tensor-core backward (bf16 inputs, fp32 gradients) against the fp64 backward oracle.

DIFF V1 with d = 64 and DIFF V2 with d = 128.  The oracle (oracle.diff_attn_v1_backward,
oracle.diff_attn_v2_backward: the chain rule of the forward with explicit maps, pinned to autograd
and to finite differences) runs on the exact values of the same bf16 inputs.  Bar: every gradient
within 2e-2 max(1, max |ref|) element by element: the kernels round P, dS, Pc and dO to bf16 for
the tensor cores (relative 2^-9 each) and sum up to n of them in fp32.
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


V1 = [  # B, H, n, causal, lambda, gamma
    (1, 1, 1, True, 0.35, True),       # one token
    (2, 2, 200, True, 0.35, True),     # two key and query tiles, ragged
    (1, 2, 300, False, -0.3, False),   # non-causal, lambda < 0, no gamma
    (1, 1, 1100, True, 1.2, True),     # nine tiles, lambda > 1
    (2, 4, 257, True, 0.6, True),      # a one-token last tile
]


@pytest.mark.parametrize("B,H,n,causal,lam,gamma", V1)
def test_v1_backward_bf16(B, H, n, causal, lam, gamma):
    d = 64
    g = torch.Generator(device="cuda").manual_seed(700 + n + H)
    x = {k: _rnd(g, B, n, H, d) for k in ("q1", "q2", "k1", "k2")}
    x["v"], x["dy"] = _rnd(g, B, n, H, 2 * d), _rnd(g, B, n, H, 2 * d)
    gam = (0.9 + 0.2 * torch.rand(2 * d, generator=g, device="cuda")) if gamma else None
    lam_t = torch.tensor([lam], device="cuda")
    got = da.diffattn_backward(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], lam_t, 0.3, x["dy"], gamma=gam,
                               causal=causal)
    da.device_status()
    ref = oracle.diff_attn_v1_backward(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], lam, 0.3,
                                       None if gam is None else gam.cpu(), 1e-5, causal, x["dy"])
    for k in ("dq1", "dq2", "dk1", "dk2", "dv"):
        _close(got[k], ref[k], k)
    _close(got["dlam"][0], ref["dlam"], "dlambda")
    if gamma:
        _close(got["dgamma"], ref["dgamma"], "dgamma")


V2 = [  # B, Hq, Hkv, n, causal, logit granularity
    (2, 4, 2, 200, True, "token"),
    (1, 8, 2, 300, True, "pair"),     # two head pairs per KV head: dK, dV summed over both
    (2, 4, 2, 129, False, "seq"),
    (1, 4, 2, 1, True, "token"),      # one token
]


@pytest.mark.parametrize("B,Hq,Hkv,n,causal,gran", V2)
def test_v2_backward_bf16(B, Hq, Hkv, n, causal, gran):
    d, G = 128, Hq // 2
    g = torch.Generator(device="cuda").manual_seed(800 + n + Hq)
    q, k, v, dy = _rnd(g, B, n, Hq, d), _rnd(g, B, n, Hkv, d), _rnd(g, B, n, Hkv, d), _rnd(g, B, n, G, d)
    shape = {"token": (B, n, G), "seq": (B, G), "pair": (G,)}[gran]
    lg = torch.randn(shape, generator=g, device="cuda")
    got = da.diffattn_v2_backward(q, k, v, lg, dy, causal=causal)
    da.device_status()
    lg_np = lg.cpu().double().numpy()
    dense = {"token": lambda: lg_np, "seq": lambda: np.broadcast_to(lg_np[:, None, :], (B, n, G)),
             "pair": lambda: np.broadcast_to(lg_np, (B, n, G))}[gran]()
    ref = oracle.diff_attn_v2_backward(q, k, v, np.ascontiguousarray(dense), causal, dy)
    dl = ref["dlogits"]
    if gran == "seq":
        dl = dl.sum(axis=1)
    elif gran == "pair":
        dl = dl.sum(axis=(0, 1))
    for key in ("dq", "dk", "dv"):
        _close(got[key], ref[key], key)
    _close(got["dlogits"], dl, "dlogits")


def test_v1_backward_bf16_bench_size_sampled_heads():
    """B4 H16 n2048 d64 causal (the bench's backward workload): per-head gradients of two heads of
    the first and last sequences against the oracle run on those heads alone; dlambda and dgamma
    (sums over every head) are finite."""
    B, H, n, d = 4, 16, 2048, 64
    g = torch.Generator(device="cuda").manual_seed(901)
    x = {k: _rnd(g, B, n, H, d) for k in ("q1", "q2", "k1", "k2")}
    x["v"], x["dy"] = _rnd(g, B, n, H, 2 * d), _rnd(g, B, n, H, 2 * d)
    gam = torch.ones(2 * d, device="cuda")
    lam = torch.tensor([0.3], device="cuda")
    got = da.diffattn_backward(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], lam, 0.2, x["dy"], gamma=gam)
    da.device_status()
    assert all(bool(torch.isfinite(t).all()) for t in got.values())
    for b in (0, B - 1):
        for h in (0, H - 1):
            sel = {k: t[b:b + 1, :, h:h + 1] for k, t in x.items()}
            ref = oracle.diff_attn_v1_backward(sel["q1"], sel["q2"], sel["k1"], sel["k2"], sel["v"], 0.3, 0.2,
                                               gam.cpu(), 1e-5, True, sel["dy"])
            for k in ("dq1", "dq2", "dk1", "dk2", "dv"):
                _close(got[k][b:b + 1, :, h:h + 1], ref[k], f"{k} b{b} h{h}")


def test_v2_backward_bf16_bench_size_sampled_pair():
    """B2 Hq32 Hkv16 n2048 d128 causal, one logit per pair: KV head 0 and 15 (with their pairs) of
    both sequences against the oracle run on that group alone."""
    B, Hq, Hkv, n, d = 2, 32, 16, 2048, 128
    G = Hq // 2
    g = torch.Generator(device="cuda").manual_seed(902)
    q, k, v, dy = _rnd(g, B, n, Hq, d), _rnd(g, B, n, Hkv, d), _rnd(g, B, n, Hkv, d), _rnd(g, B, n, G, d)
    lg = torch.randn((G,), generator=g, device="cuda")
    got = da.diffattn_v2_backward(q, k, v, lg, dy)
    da.device_status()
    assert all(bool(torch.isfinite(t).all()) for t in got.values())
    for b in (0, B - 1):
        for hk in (0, Hkv - 1):
            qs = q[b:b + 1, :, 2 * hk:2 * hk + 2]
            ks, vs = k[b:b + 1, :, hk:hk + 1], v[b:b + 1, :, hk:hk + 1]
            lgs = np.broadcast_to(lg[hk:hk + 1].cpu().double().numpy(), (1, n, 1))
            ref = oracle.diff_attn_v2_backward(qs, ks, vs, np.ascontiguousarray(lgs), True, dy[b:b + 1, :, hk:hk + 1])
            _close(got["dq"][b:b + 1, :, 2 * hk:2 * hk + 2], ref["dq"], f"dq b{b} kv{hk}")
            _close(got["dk"][b:b + 1, :, hk:hk + 1], ref["dk"], f"dk b{b} kv{hk}")
            _close(got["dv"][b:b + 1, :, hk:hk + 1], ref["dv"], f"dv b{b} kv{hk}")


def test_v1_backward_bench_size_cross_head_sums():
    """dlambda and dgamma are sums over every (sequence, head, row); at B4 H16 n2048 d64 the fp32
    path gathers them from hundreds of row-pass blocks and the tensor-core path from its
    statistics-pass blocks.  Both are compared with the sum of the oracle's per-head gradients over
    all 64 heads, on the same bf16-exact inputs (fed to the fp32 path as fp32).  Bar: the path's
    element tolerance (1e-4 fp32, 2e-2 bf16) times max(1, sum over heads of |per-head value|), the
    magnitude the accumulation runs through."""
    B, H, n, d = 4, 16, 2048, 64
    g = torch.Generator(device="cuda").manual_seed(903)
    x = {k: _rnd(g, B, n, H, d) for k in ("q1", "q2", "k1", "k2")}
    x["v"], x["dy"] = _rnd(g, B, n, H, 2 * d), _rnd(g, B, n, H, 2 * d)
    gam = 0.9 + 0.2 * torch.rand(2 * d, generator=g, device="cuda")
    lam, lin = 0.3, 0.2
    lam_t = torch.tensor([lam], device="cuda")
    got = {"bf16": da.diffattn_backward(*(x[k] for k in ("q1", "q2", "k1", "k2", "v")), lam_t, lin, x["dy"],
                                        gamma=gam)}
    xf = {k: t.float() for k, t in x.items()}
    got["f32"] = da.diffattn_backward(*(xf[k] for k in ("q1", "q2", "k1", "k2", "v")), lam_t, lin, xf["dy"],
                                      gamma=gam)
    da.device_status()
    dlam, dlam_abs = 0.0, 0.0
    dgam, dgam_abs = np.zeros(2 * d), np.zeros(2 * d)
    gam_np = gam.cpu()
    xc = {k: t.cpu() for k, t in x.items()}
    for b in range(B):
        for h in range(H):
            sel = {k: t[b:b + 1, :, h:h + 1] for k, t in xc.items()}
            ref = oracle.diff_attn_v1_backward(sel["q1"], sel["q2"], sel["k1"], sel["k2"], sel["v"], lam, lin,
                                               gam_np, 1e-5, True, sel["dy"])
            dlam += float(ref["dlam"])
            dlam_abs += abs(float(ref["dlam"]))
            dgam += np.asarray(ref["dgamma"], np.float64)
            dgam_abs += np.abs(np.asarray(ref["dgamma"], np.float64))
    for dt, tol in (("f32", 1e-4), ("bf16", 2e-2)):
        e_lam = abs(float(got[dt]["dlam"][0]) - dlam)
        assert e_lam <= tol * max(1.0, dlam_abs), f"{dt} dlambda: {e_lam} vs {dlam} (sum |.| {dlam_abs})"
        e_gam = np.abs(got[dt]["dgamma"].cpu().double().numpy() - dgam)
        assert np.all(e_gam <= tol * np.maximum(1.0, dgam_abs)), f"{dt} dgamma: max {float(e_gam.max())}"
