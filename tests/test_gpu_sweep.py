"""Seeded sweep of small shapes through the bf16 tensor-core paths, full compare against the oracle.

Shapes are drawn from a fixed seed so that every run checks the same cases: batch, heads, sequence
lengths across tile boundaries (1 .. 700, including exact multiples of 128 and one past them), both
head widths, causal and not, lambda below 0, inside [0, 1] and above 1, and GQA groups of 2 and 4
for DIFF V2.  Each case compares every output element with the fp64 oracle at the operator's bar
(2e-2 absolute on the normalised bf16 output; DIFF V2 at 2e-2 max(1, max |ref|)).  The decode step is
swept the same way over cache lengths and ragged per-sequence lengths.
"""

import numpy as np
import pytest
import torch

import oracle
from differential_attention_03_gb300 import binding as da

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    from differential_attention_03_gb300 import build
    build.build()
    torch.cuda.init()


def _cases(seed, count, draw):
    rng = np.random.default_rng(seed)
    return [draw(rng) for _ in range(count)]


def _n(rng):
    return int(rng.choice([1, 2, 127, 128, 129, 255, 256, 257, int(rng.integers(3, 700))]))


V1_CASES = _cases(2024, 10, lambda r: (int(r.integers(1, 3)), int(r.integers(1, 4)), _n(r), int(r.choice([64, 128])),
                                       bool(r.integers(0, 2)), float(r.choice([-0.4, 0.3, 0.8, 1.3]))))


@pytest.mark.parametrize("B,H,n,d,causal,lam", V1_CASES)
def test_v1_forward_sweep(B, H, n, d, causal, lam):
    g = torch.Generator(device="cuda").manual_seed(B * 7919 + H * 131 + n * 17 + d)
    x = {k: torch.randn((B, n, H, d), generator=g, device="cuda").to(torch.bfloat16) for k in ("q1", "q2", "k1", "k2")}
    x["v"] = torch.randn((B, n, H, 2 * d), generator=g, device="cuda").to(torch.bfloat16)
    gam = 0.9 + 0.2 * torch.rand(2 * d, generator=g, device="cuda")
    lin = da.lambda_init(3)
    out = da.diffattn_forward(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], torch.tensor([lam], device="cuda"), lin,
                              gamma=gam, causal=causal)
    da.device_status()
    ref = oracle.diff_attn_v1(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], lam, oracle.lambda_init(3), gam.cpu(), 1e-5,
                              causal)
    err = float(np.max(np.abs(out.float().cpu().double().numpy() - ref)))
    assert err <= TOL, f"max abs error {err}"


V2_CASES = _cases(2025, 8, lambda r: (int(r.integers(1, 3)), int(r.choice([2, 4])), _n(r), bool(r.integers(0, 2))))


@pytest.mark.parametrize("B,Hkv,n,causal", V2_CASES)
def test_v2_forward_sweep(B, Hkv, n, causal):
    d = 128
    grp = 2 if Hkv == 4 else 4  # query heads per KV head
    Hq = Hkv * grp
    g = torch.Generator(device="cuda").manual_seed(B * 104729 + Hkv * 31 + n)
    q = torch.randn((B, n, Hq, d), generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn((B, n, Hkv, d), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((B, n, Hkv, d), generator=g, device="cuda").to(torch.bfloat16)
    lg = torch.randn((B, n, Hq // 2), generator=g, device="cuda")
    out = da.diffattn_v2_forward(q, k, v, lg, causal=causal)
    da.device_status()
    ref = oracle.diff_attn_v2(q, k, v, lg.cpu().double().numpy(), causal)
    err = float(np.max(np.abs(out.float().cpu().double().numpy() - ref)))
    assert err <= TOL * max(1.0, float(np.max(np.abs(ref)))), f"max abs error {err}"


DEC_CASES = _cases(2026, 8, lambda r: (int(r.integers(1, 5)), int(r.integers(1, 4)), int(r.integers(1, 3000)),
                                       int(r.choice([64, 128])), bool(r.integers(0, 2))))


@pytest.mark.parametrize("B,H,n,d,ragged", DEC_CASES)
def test_v1_decode_sweep(B, H, n, d, ragged):
    g = torch.Generator(device="cuda").manual_seed(B * 65537 + H * 257 + n + d)
    q1, q2 = (torch.randn((B, H, d), generator=g, device="cuda").to(torch.bfloat16) for _ in range(2))
    k1, k2 = (torch.randn((B, n, H, d), generator=g, device="cuda").to(torch.bfloat16) for _ in range(2))
    v = torch.randn((B, n, H, 2 * d), generator=g, device="cuda").to(torch.bfloat16)
    lens = None
    if ragged:
        lens = torch.randint(0, n + 1, (B,), generator=torch.Generator().manual_seed(n), dtype=torch.int32)
    lam = torch.tensor([0.45], device="cuda")
    lin = da.lambda_init(5)
    out = da.diffattn_decode(q1, q2, k1, k2, v, lam, lin, lens=None if lens is None else lens.cuda())
    da.device_status()
    ref = oracle.diff_attn_v1_decode(q1, q2, k1, k2, v, 0.45, oracle.lambda_init(5), None, 1e-5,
                                     None if lens is None else lens.numpy())
    err = float(np.max(np.abs(out.float().cpu().double().numpy() - ref)))
    assert err <= TOL, f"max abs error {err}"
