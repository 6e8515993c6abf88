"""CUDA-graph capture of the entry points.

Every device entry point is asynchronous on the caller's stream, allocates nothing and never
synchronises, so a serving loop (one decode step per layer and token) or a training step can capture
its calls once and replay them with one launch.  Each case here runs the calls eagerly first (the
library's one-time set-up: the tensor-map encoder and the status word), captures them on a side
stream, then copies new inputs into the captured buffers and replays: the replay's outputs must equal
those of eager calls on the same new inputs bit for bit (the same kernels on the same data); only dQ
of the backward, which is summed by reduce-adds in whatever order they land, is compared to 1e-5.
"""

import pytest
import torch

from differential_attention_03_gb300 import binding as da

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from differential_attention_03_gb300 import build
    build.build()
    torch.cuda.init()


def _capture(fn):
    """Warm fn up on a side stream, then capture one call of it; returns (graph, captured outputs)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    da.device_status()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = fn()
    return g, out


def _refill(gen, *tensors):
    for t in tensors:
        t.copy_(torch.randn(t.shape, generator=gen, device="cuda").to(t.dtype))


def _bf16(gen, *shape):
    return torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16)


@pytest.mark.parametrize("d,n", [(64, 700), (128, 300), (64, 9000)])
def test_graph_v1_lambda_and_forward(d, n):
    # lambda_reparam and the forward of one layer in one graph (n = 9000 at d = 64: one CTA per item)
    B, H = 2, 3
    g = torch.Generator(device="cuda").manual_seed(d + n)
    x = {k: _bf16(g, B, n, H, d) for k in ("q1", "q2", "k1", "k2")}
    v = _bf16(g, B, n, H, 2 * d)
    lv = [0.1 * torch.randn(d, generator=g, device="cuda") for _ in range(4)]
    gamma = 0.9 + 0.2 * torch.rand(2 * d, generator=g, device="cuda")
    lam = torch.empty(1, device="cuda")
    out = torch.empty_like(v)
    lin = da.lambda_init(5)

    def step():
        da.lambda_reparam(*lv, lin, out=lam)
        return da.diffattn_forward(x["q1"], x["q2"], x["k1"], x["k2"], v, lam, lin, gamma=gamma, out=out)

    graph, captured = _capture(step)
    for it in range(3):
        _refill(g, *x.values(), v, *lv)
        graph.replay()
        lam_e = da.lambda_reparam(*lv, lin)
        ref = da.diffattn_forward(x["q1"], x["q2"], x["k1"], x["k2"], v, lam_e, lin, gamma=gamma)
        torch.cuda.synchronize()
        da.device_status()
        assert torch.equal(lam, lam_e)
        assert torch.equal(captured, ref), f"replay {it}"


def test_graph_v2_forward():
    B, Hq, Hkv, n, d = 2, 8, 4, 513, 128
    g = torch.Generator(device="cuda").manual_seed(11)
    q, k, v = _bf16(g, B, n, Hq, d), _bf16(g, B, n, Hkv, d), _bf16(g, B, n, Hkv, d)
    lg = torch.randn((B, n, Hq // 2), generator=g, device="cuda")
    out = torch.empty((B, n, Hq // 2, d), device="cuda", dtype=torch.bfloat16)
    graph, captured = _capture(lambda: da.diffattn_v2_forward(q, k, v, lg, out=out))
    for it in range(2):
        _refill(g, q, k, v, lg)
        graph.replay()
        ref = da.diffattn_v2_forward(q, k, v, lg)
        torch.cuda.synchronize()
        da.device_status()
        assert torch.equal(captured, ref), f"replay {it}"


def test_graph_decode_steps_of_several_layers():
    # Eight decode calls (eight layers' caches) in one graph, with per-sequence lengths that change
    # between replays; the last two layers use the allocation-free entry point.
    B, H, n, d, layers = 3, 4, 2000, 64, 8
    g = torch.Generator(device="cuda").manual_seed(12)
    cache = [{"k1": _bf16(g, B, n, H, d), "k2": _bf16(g, B, n, H, d), "v": _bf16(g, B, n, H, 2 * d)}
             for _ in range(layers)]
    q = [(_bf16(g, B, H, d), _bf16(g, B, H, d)) for _ in range(layers)]
    lam = torch.tensor([0.4], device="cuda")
    lens = torch.tensor([n, 1, 777], dtype=torch.int32, device="cuda")
    ws = torch.empty(da.decode_workspace_bytes(B, H, d), dtype=torch.uint8, device="cuda")
    outs = [torch.empty((B, H, 2 * d), device="cuda", dtype=torch.bfloat16) for _ in range(layers)]

    def call(i, out=None):
        c = cache[i]
        if i >= layers - 2:
            return da.diffattn_decode_noalloc(q[i][0], q[i][1], c["k1"], c["k2"], c["v"], lam, 0.2, lens=lens,
                                              out=out)
        return da.diffattn_decode(q[i][0], q[i][1], c["k1"], c["k2"], c["v"], lam, 0.2, lens=lens, out=out,
                                  workspace=ws)

    def step():
        for i in range(layers):
            call(i, outs[i])
        return outs

    graph, _ = _capture(step)
    for it, new_lens in enumerate(([5, n, 1024], [0, 129, n])):
        lens.copy_(torch.tensor(new_lens, dtype=torch.int32))
        for i in range(layers):
            _refill(g, *q[i])
        graph.replay()
        refs = [call(i) for i in range(layers)]
        torch.cuda.synchronize()
        da.device_status()
        for i in range(layers):
            assert torch.equal(outs[i], refs[i]), f"replay {it}, layer {i}"


def test_graph_backward():
    B, H, n, d = 2, 2, 600, 64
    g = torch.Generator(device="cuda").manual_seed(13)
    x = {k: _bf16(g, B, n, H, d) for k in ("q1", "q2", "k1", "k2")}
    v, dy = _bf16(g, B, n, H, 2 * d), _bf16(g, B, n, H, 2 * d)
    lam = torch.tensor([0.35], device="cuda")
    ws = torch.empty(da.backward_workspace_bytes(B, H, n, d), dtype=torch.uint8, device="cuda")

    def step():
        return da.diffattn_backward(x["q1"], x["q2"], x["k1"], x["k2"], v, lam, 0.2, dy, workspace=ws)

    graph, captured = _capture(step)
    for it in range(2):
        _refill(g, *x.values(), v, dy)
        graph.replay()
        ws_e = torch.empty_like(ws)
        ref = da.diffattn_backward(x["q1"], x["q2"], x["k1"], x["k2"], v, lam, 0.2, dy, workspace=ws_e)
        torch.cuda.synchronize()
        da.device_status()
        for k in ("dk1", "dk2", "dv", "dlam", "dgamma"):
            assert torch.equal(captured[k], ref[k]), f"replay {it}: {k}"
        for k in ("dq1", "dq2"):
            err = float((captured[k] - ref[k]).abs().max())
            assert err <= 1e-5 * max(1.0, float(ref[k].abs().max())), f"replay {it}: {k} {err}"


@pytest.mark.parametrize("B,n", [(1, 2000), (3, 300)])
def test_graph_host_buffer_forward(B, n):
    # diffattn_forward_host forks its copies and (token-range) forwards onto internal streams with
    # events and joins them back into the caller's stream, which stream capture records as a fork
    # and join: the graph holds the host->device copies, the forwards and the copies back.  New
    # inputs written into the same page-locked buffers are picked up by the next replay.
    H, d = 2, 128
    g = torch.Generator(device="cuda").manual_seed(14 + n)
    host = {k: torch.empty((B, n, H, d), dtype=torch.bfloat16).pin_memory() for k in ("q1", "q2", "k1", "k2")}
    host["v"] = torch.empty((B, n, H, 2 * d), dtype=torch.bfloat16).pin_memory()
    out = torch.empty((B, n, H, 2 * d), dtype=torch.bfloat16).pin_memory()
    lam = torch.tensor([0.45], device="cuda")
    ws = torch.empty(da.forward_host_workspace_bytes(torch.bfloat16, B, H, n, d), dtype=torch.uint8, device="cuda")

    def fill():
        for t in host.values():
            t.copy_(torch.randn(t.shape, generator=g, device="cuda").to(torch.bfloat16).cpu())

    fill()
    graph, _ = _capture(lambda: da.diffattn_forward_host(host["q1"], host["q2"], host["k1"], host["k2"], host["v"],
                                                         lam, 0.2, out=out, workspace=ws))
    for it in range(2):
        fill()
        graph.replay()
        torch.cuda.synchronize()
        dev = {k: t.cuda() for k, t in host.items()}
        ref = da.diffattn_forward(dev["q1"], dev["q2"], dev["k1"], dev["k2"], dev["v"], lam, 0.2)
        torch.cuda.synchronize()
        da.device_status()
        assert torch.equal(out, ref.cpu()), f"replay {it}"
