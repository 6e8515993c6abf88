"""GPU parity of the projections and of the attention layers around the operator.

The projection GEMM is compared with an fp64 matrix product of the same bf16
inputs: the kernel accumulates in fp32 and rounds once to bf16, so each
element is within 2^-8 |ref| (twice the bf16 half-ulp) plus 1e-5 sum_k |a_k
w_k| (fp32 accumulation) of it.

The layers are compared with the fp64 layer oracle (oracle.diff_v1_layer,
oracle.diff_v2_layer).  Their inputs are drawn so that every projection is
exact in bf16: X has a few entries of +-1 per row and W^Q, W^K, W^V,
W^lambda hold small multiples of 1/4 or 1/8, so X W is a short sum of
multiples of 1/8 that fp32 accumulates and bf16 stores without rounding.
Then the projections in the workspace must equal the fp64 products bit for
bit, the normalised heads y must meet the operator's own bar (2e-2), and
the output out = y W^O (W^O with a few +-1/8 entries per row) is within
2e-2 ||W^O_j||_1 + 2^-8 |ref| of the oracle: the operator's bar carried
through W^O, plus the bf16 rounding of out.
"""

import numpy as np
import pytest
import torch

import oracle
from differential_attention_03_gb300 import binding as da

pytestmark = pytest.mark.gpu

OP_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    from differential_attention_03_gb300 import build
    build.build()
    torch.cuda.init()


def _f64(t):
    return t.detach().float().cpu().double().numpy()


# ----------------------------------------------------------------------------- projection
@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (130, 264, 72), (300, 520, 200), (1000, 768, 3072),
                                   (257, 9216, 3072)])
def test_projection_matches_fp64_product(M, N, K):
    g = torch.Generator(device="cuda").manual_seed(M + N + K)
    a = torch.randn((M, K), generator=g, device="cuda").to(torch.bfloat16)
    w = torch.randn((N, K), generator=g, device="cuda").to(torch.bfloat16)
    out = da.projection(a, w)
    da.device_status()
    A, W = _f64(a), _f64(w)
    ref = A @ W.T
    bound = 2.0 ** -8 * np.abs(ref) + 1e-5 * (np.abs(A) @ np.abs(W).T)
    err = np.abs(_f64(out) - ref)
    assert np.all(err <= bound), float(np.max(err - bound))


def test_projection_large_sampled_rows():
    """A 8192 x 9216 x 3072 product (a C3-sized X [W^Q | W^K | W^V]) on sampled rows."""
    M, N, K = 8192, 9216, 3072
    g = torch.Generator(device="cuda").manual_seed(7)
    a = torch.randn((M, K), generator=g, device="cuda").to(torch.bfloat16)
    w = torch.randn((N, K), generator=g, device="cuda").to(torch.bfloat16)
    out = da.projection(a, w)
    da.device_status()
    rows = np.unique(np.concatenate([[0, 127, 128, M - 1], np.random.default_rng(1).integers(0, M, 24)]))
    A, W = _f64(a[rows]), _f64(w)
    ref = A @ W.T
    bound = 2.0 ** -8 * np.abs(ref) + 1e-5 * (np.abs(A) @ np.abs(W).T)
    err = np.abs(_f64(out[rows]) - ref)
    assert np.all(err <= bound)


# ----------------------------------------------------------------------------- layers
def _sparse_signs(rng, rows, cols, per_row, scale=1.0):
    """rows x cols with `per_row` entries of +-scale per row, zeros elsewhere."""
    x = np.zeros((rows, cols))
    for r in range(rows):
        idx = rng.choice(cols, size=per_row, replace=False)
        x[r, idx] = scale * rng.choice([-1.0, 1.0], size=per_row)
    return x


def _small_multiples(rng, shape, lo, hi, unit):
    return rng.integers(lo, hi + 1, size=shape) * unit


def _bf16(a, device="cuda"):
    t = torch.tensor(np.ascontiguousarray(a), dtype=torch.float64).to(torch.bfloat16)
    assert np.array_equal(t.double().numpy(), a), "input not exact in bf16"
    return t.to(device)


@pytest.mark.parametrize("B,n,D,H,d,causal", [(2, 200, 256, 2, 64, True), (1, 333, 512, 2, 128, True),
                                              (2, 150, 256, 2, 64, False), (1, 129, 384, 1, 128, False)])
def test_v1_layer_matches_oracle(B, n, D, H, d, causal):
    rng = np.random.default_rng(B * 1000 + n + d)
    x = _sparse_signs(rng, B * n, D, 8).reshape(B, n, D)
    wq, wk = (_small_multiples(rng, (D, H * 2 * d), -4, 4, 0.25) for _ in range(2))
    wv = _small_multiples(rng, (D, H * 2 * d), -2, 2, 0.125)
    wo = _sparse_signs(rng, D, H * 2 * d, 8, 0.125).T  # [H 2d, D]: column j of W^O has 8 entries
    lam_vecs = [rng.normal(0, 0.1, d) for _ in range(4)]
    gamma = rng.uniform(0.9, 1.1, 2 * d)
    lin = oracle.lambda_init(3)

    xt = _bf16(x)
    w_qkv = _bf16(np.concatenate([wq.T, wk.T, wv.T], axis=0))
    w_o = _bf16(np.ascontiguousarray(wo.T))
    lv = [torch.tensor(v, dtype=torch.float32, device="cuda") for v in lam_vecs]
    gt = torch.tensor(gamma, dtype=torch.float32, device="cuda")
    ws = torch.empty(da.layer_workspace_bytes(B, n, H, d), dtype=torch.uint8, device="cuda")
    out = da.layer_forward(xt, w_qkv, w_o, *lv, lin, H, gamma=gt, causal=causal, workspace=ws)
    da.device_status()

    M = B * n
    # 1. the fused projection, read back from the workspace, is exact
    qkv = ws[: M * 6 * H * d * 2].view(torch.bfloat16).view(M, 6 * H * d)
    ref_qkv = x.reshape(M, D) @ np.concatenate([wq, wk, wv], axis=1)
    assert np.array_equal(_f64(qkv), ref_qkv)
    # 2. the normalised heads meet the operator's bar
    off = (M * 6 * H * d * 2 + 255) // 256 * 256
    y = ws[off: off + M * 2 * H * d * 2].view(torch.bfloat16).view(B, n, H, 2 * d)
    q = ref_qkv[:, : 2 * H * d].reshape(B, n, H, 2 * d)
    k = ref_qkv[:, 2 * H * d: 4 * H * d].reshape(B, n, H, 2 * d)
    v = ref_qkv[:, 4 * H * d:].reshape(B, n, H, 2 * d)
    lam = oracle.lambda_reparam(*lam_vecs, lin)
    ref_y = oracle.diff_attn_v1(q[..., :d], q[..., d:], k[..., :d], k[..., d:], v, lam, lin, gamma, 1e-5, causal)
    assert float(np.max(np.abs(_f64(y) - ref_y))) <= OP_TOL
    # 3. the layer output against the layer oracle, the bar carried through W^O
    ref = oracle.diff_v1_layer(x, wq, wk, wv, wo, *lam_vecs, lin, H, gamma, 1e-5, causal)
    bound = OP_TOL * np.abs(wo).sum(axis=0) + 2.0 ** -8 * np.abs(ref)
    assert np.all(np.abs(_f64(out) - ref) <= bound)


@pytest.mark.parametrize("B,n,D,Hq,Hkv,causal", [(2, 200, 256, 4, 2, True), (1, 300, 512, 8, 2, True),
                                                 (1, 129, 256, 4, 2, False)])
def test_v2_layer_matches_oracle(B, n, D, Hq, Hkv, causal):
    d, G = 128, Hq // 2
    rng = np.random.default_rng(B * 77 + n + Hq)
    x = _sparse_signs(rng, B * n, D, 8).reshape(B, n, D)
    wq = _small_multiples(rng, (D, Hq * d), -4, 4, 0.25)
    wk = _small_multiples(rng, (D, Hkv * d), -4, 4, 0.25)
    wv = _small_multiples(rng, (D, Hkv * d), -2, 2, 0.125)
    wl = _small_multiples(rng, (D, G), -2, 2, 0.125)
    wo = _sparse_signs(rng, D, G * d, 8, 0.125).T  # [G d, D]

    xt = _bf16(x)
    w_qkvl = _bf16(np.concatenate([wq.T, wk.T, wv.T, wl.T], axis=0))
    w_o = _bf16(np.ascontiguousarray(wo.T))
    ws = torch.empty(da.v2_layer_workspace_bytes(B, n, Hq, Hkv, d), dtype=torch.uint8, device="cuda")
    out = da.v2_layer_forward(xt, w_qkvl, w_o, Hq, Hkv, causal=causal, workspace=ws)
    da.device_status()

    M, nq = B * n, (Hq + 2 * Hkv) * d
    r256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    qkv = ws[: M * nq * 2].view(torch.bfloat16).view(M, nq)
    logits = ws[r256(M * nq * 2): r256(M * nq * 2) + M * G * 4].view(torch.float32).view(M, G)
    xm = x.reshape(M, D)
    assert np.array_equal(_f64(qkv), xm @ np.concatenate([wq, wk, wv], axis=1))
    assert np.array_equal(logits.cpu().double().numpy(), xm @ wl)
    ref = oracle.diff_v2_layer(x, wq, wk, wv, wl, wo, Hq, Hkv, causal)
    bound = OP_TOL * np.abs(wo).sum(axis=0) + 2.0 ** -8 * np.abs(ref)
    assert np.all(np.abs(_f64(out) - ref) <= bound)


def test_v1_layer_reads_projections_like_the_contiguous_path():
    """At a 3B-shaped size (D 3072, H 12, d 128) the layer, which reads Q_1 .. V in place through
    strided tensor maps, gives the same bits as the projection, a copy into contiguous tensors,
    diffattn_forward and the W^O projection called one by one."""
    B, n, D, H, d = 1, 1024, 3072, 12, 128
    g = torch.Generator(device="cuda").manual_seed(31)
    x = torch.randn((B, n, D), generator=g, device="cuda").to(torch.bfloat16)
    w_qkv = (torch.randn((6 * H * d, D), generator=g, device="cuda") / D ** 0.5).to(torch.bfloat16)
    w_o = (torch.randn((D, 2 * H * d), generator=g, device="cuda") / (2 * H * d) ** 0.5).to(torch.bfloat16)
    lv = [0.1 * torch.randn(d, generator=g, device="cuda") for _ in range(4)]
    lin = da.lambda_init(12)
    out = da.layer_forward(x, w_qkv, w_o, *lv, lin, H)
    qkv = da.projection(x.view(B * n, D), w_qkv).view(B, n, 3, H, 2 * d)
    q1, q2 = qkv[:, :, 0, :, :d].contiguous(), qkv[:, :, 0, :, d:].contiguous()
    k1, k2 = qkv[:, :, 1, :, :d].contiguous(), qkv[:, :, 1, :, d:].contiguous()
    v = qkv[:, :, 2].contiguous()
    lam = da.lambda_reparam(*lv, lin)
    y = da.diffattn_forward(q1, q2, k1, k2, v, lam, lin)
    ref = da.projection(y.view(B * n, 2 * H * d), w_o).view(B, n, D)
    da.device_status()
    assert torch.equal(out, ref)
