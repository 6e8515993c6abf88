"""The decode step for callers that cannot allocate device memory.

diffattn_decode_noalloc takes no workspace: the partial states of the
clusters that share a (batch, head) pair's keys go to a fixed scratch array
inside the library, for callers such as a plugin whose host framework owns
all device memory, or a serving loop that may not call cudaMalloc after
start-up.  This test calls it through the C ABI and compares its output with
diffattn_decode given a caller-allocated workspace (the same split), within
the bf16 parity bar, on two calls in a row with different inputs and lengths:
the second call must not see anything the first left in the shared scratch.

The file name sorts last so that a run stopping at the first failure has run
every other test first; it also passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

from differential_attention_03_gb300 import binding as da
from differential_attention_03_gb300 import build

pytestmark = pytest.mark.gpu

TOL = 2e-2  # the bf16 parity bar (max abs error on the normalised output)


def _inputs(B, H, n, d, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)

    def rnd(*shape, std=1.0):
        return (std * torch.randn(shape, generator=g, device="cuda", dtype=torch.float32)).to(torch.bfloat16)
    x = {"q1": rnd(B, H, d), "q2": rnd(B, H, d), "k1": rnd(B, n, H, d), "k2": rnd(B, n, H, d),
         "v": rnd(B, n, H, 2 * d)}
    x["gamma"] = 0.9 + 0.2 * torch.rand(2 * d, generator=g, device="cuda")
    x["lam"] = torch.tensor([0.35], device="cuda")
    return x


def _noalloc_via_abi(L, x, lin, lens, out):
    B, n, H, d = x["k1"].shape
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = L.diffattn_decode_noalloc(da.BF16, B, H, n, d, p(x["q1"]), p(x["q2"]), p(x["k1"]), p(x["k2"]),
                                   p(x["v"]), p(lens), p(x["lam"]), ctypes.c_float(lin), p(x["gamma"]),
                                   ctypes.c_float(1e-5), p(out),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == da.OK, L.diffattn_last_error()


@pytest.mark.parametrize("B,H,n,d,lens_pair", [
    (1, 16, 8192, 64, (None, [5000])),          # few pairs: split over clusters
    (2, 3, 9000, 128, ([9000, 2500], [1, 8191])),
])
def test_decode_noalloc_matches_workspace_decode(B, H, n, d, lens_pair):
    build.build()
    L = da.lib()
    lin = 0.55
    for call, lens in enumerate(lens_pair):
        x = _inputs(B, H, n, d, seed=500 + 10 * call + d)
        lens_t = None if lens is None else torch.tensor(lens * (B // len(lens)), dtype=torch.int32,
                                                        device="cuda")
        ws = torch.empty(da.decode_workspace_bytes(B, H, d), dtype=torch.uint8, device="cuda")
        ref = da.diffattn_decode(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], x["lam"], lin, gamma=x["gamma"],
                                 lens=lens_t, workspace=ws)
        out = torch.full((B, H, 2 * d), float("nan"), device="cuda", dtype=torch.bfloat16)
        _noalloc_via_abi(L, x, lin, lens_t, out)
        da.device_status()
        err = float(np.max(np.abs(out.float().cpu().numpy() - ref.float().cpu().numpy())))
        assert err <= TOL, (call, err)
