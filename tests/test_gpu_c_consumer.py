"""The C ABI from a plain C program: no PyTorch in the process, only diffattn.h and the CUDA runtime.

`tests/c/abi_consumer.c` is compiled with gcc against include/diffattn.h and the in-tree
libdiffattn.so, reads seeded inputs from a file, runs lambda_reparam, the bf16 forward and the bf16
decode step on one stream, reads the device status word and writes the results.  This test writes
the inputs (numpy, seeded), runs the program and compares its outputs with the oracle: lambda to
1e-6, the forward and the decode step at the 2e-2 bar of the bf16 path.
"""

import glob
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TOL = 2e-2


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16, as raw 16-bit words."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def _bf16_values(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _cudart_dir():
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    for pat in ("lib64/libcudart.so", "targets/*/lib/libcudart.so", "lib/libcudart.so"):
        hits = glob.glob(os.path.join(home, pat))
        if hits:
            return home, os.path.dirname(hits[0])
    pytest.skip("libcudart.so not found")


@pytest.fixture(scope="module")
def consumer(tmp_path_factory):
    from differential_attention_03_gb300 import build
    lib = build.build()
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    home, libdir = _cudart_dir()
    exe = str(tmp_path_factory.mktemp("c") / "abi_consumer")
    pkg = os.path.dirname(lib)
    cmd = ["gcc", "-std=c99", "-O2", "-Wall", "-I", os.path.join(ROOT, "include"), "-I",
           os.path.join(home, "include"), os.path.join(ROOT, "tests", "c", "abi_consumer.c"), "-o", exe,
           "-L", pkg, "-ldiffattn", "-L", libdir, "-lcudart", f"-Wl,-rpath,{pkg}", f"-Wl,-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


@pytest.mark.parametrize("B,H,n,d,nc,causal", [(2, 3, 300, 64, 1000, 1), (1, 2, 129, 128, 513, 0)])
def test_c_consumer_matches_oracle(consumer, tmp_path, B, H, n, d, nc, causal):
    rng = np.random.default_rng(1000 + n + d)
    layer = 3
    lin = oracle.lambda_init(layer)
    bits = {k: _bf16_bits(rng.standard_normal(s)) for k, s in (
        ("q1", (B, n, H, d)), ("q2", (B, n, H, d)), ("k1", (B, n, H, d)), ("k2", (B, n, H, d)),
        ("v", (B, n, H, 2 * d)), ("tq1", (B, H, d)), ("tq2", (B, H, d)), ("tk1", (B, nc, H, d)),
        ("tk2", (B, nc, H, d)), ("tv", (B, nc, H, 2 * d)))}
    lv = {k: (0.1 * rng.standard_normal(d)).astype(np.float32) for k in ("lq1", "lk1", "lq2", "lk2")}
    gamma = (0.9 + 0.2 * rng.random(2 * d)).astype(np.float32)
    lens = np.array([nc] + [nc // 2 + 1] * (B - 1), dtype=np.int32)  # a full and a shorter cache

    inp = tmp_path / "in.bin"
    with open(inp, "wb") as f:
        f.write(np.array([B, H, n, d, nc, causal], dtype=np.int32).tobytes())
        f.write(np.float32(lin).tobytes())
        for k in ("q1", "q2", "k1", "k2", "v"):
            f.write(bits[k].tobytes())
        for k in ("lq1", "lk1", "lq2", "lk2"):
            f.write(lv[k].tobytes())
        f.write(gamma.tobytes())
        for k in ("tq1", "tq2", "tk1", "tk2", "tv"):
            f.write(bits[k].tobytes())
        f.write(lens.tobytes())
    outp = tmp_path / "out.bin"
    r = subprocess.run([consumer, str(inp), str(outp)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok")

    raw = np.fromfile(outp, dtype=np.uint8)
    lam = float(raw[:4].view(np.float32)[0])
    nout = B * n * H * 2 * d
    out = _bf16_values(raw[4:4 + 2 * nout].view(np.uint16)).reshape(B, n, H, 2 * d)
    dec = _bf16_values(raw[4 + 2 * nout:].view(np.uint16)).reshape(B, H, 2 * d)

    lam_ref = oracle.lambda_reparam(*(lv[k].astype(np.float64) for k in ("lq1", "lk1", "lq2", "lk2")), lin)
    assert abs(lam - lam_ref) <= 1e-6 * max(1.0, abs(lam_ref))
    val = {k: _bf16_values(b) for k, b in bits.items()}
    ref = oracle.diff_attn_v1(val["q1"], val["q2"], val["k1"], val["k2"], val["v"], lam, lin,
                              gamma.astype(np.float64), 1e-5, bool(causal))
    assert float(np.max(np.abs(out - ref))) <= TOL
    ref_dec = oracle.diff_attn_v1_decode(val["tq1"], val["tq2"], val["tk1"], val["tk2"], val["tv"], lam, lin,
                                         gamma.astype(np.float64), 1e-5, lens)
    assert float(np.max(np.abs(dec - ref_dec))) <= TOL
