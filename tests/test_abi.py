"""C ABI checks that need no GPU: the library builds and loads, exports every
symbol include/diffattn.h declares, and rejects bad arguments on the host
before any CUDA call (these calls never reach the device)."""

import ctypes
import glob
import os
import re
import shutil
import subprocess

import pytest

import oracle
from differential_attention_03_gb300 import binding as da
from differential_attention_03_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "diffattn.h")


@pytest.fixture(scope="module")
def L():
    build.build()
    return da.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([A-Za-z_]\w*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_is_strict_c99_and_a_c_program_links(L, tmp_path):
    # The header alone compiles as pedantic C99; the plain C consumer of the GPU tests
    # (tests/c/abi_consumer.c) compiles warning-free and links against libdiffattn.so.
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = tmp_path / "h.c"
    src.write_text('#include "diffattn.h"\nint main(void) { return (int)DIFFATTN_OK + (int)DIFFATTN_BF16 - 1; }\n')
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I",
                        os.path.join(ROOT, "include"), str(src), "-o", str(tmp_path / "h")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    libs = glob.glob(os.path.join(home, "lib64", "libcudart.so")) + glob.glob(
        os.path.join(home, "targets", "*", "lib", "libcudart.so"))
    if not libs:
        pytest.skip("libcudart.so not found")
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-I", os.path.join(home, "include"), os.path.join(ROOT, "tests", "c", "abi_consumer.c"),
                        "-o", str(tmp_path / "consumer"), "-L", os.path.dirname(build.LIB), "-ldiffattn",
                        "-L", os.path.dirname(libs[0]), "-lcudart"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_header_declares_the_entry_points():
    names = _declared()
    for want in ("diffattn_forward", "diffattn_v2_forward", "lambda_reparam", "diffattn_lambda_init",
                 "diffattn_device_status", "diffattn_last_error", "diffattn_forward_host",
                 "diffattn_forward_host_workspace", "diffattn_decode", "diffattn_v2_decode",
                 "diffattn_decode_workspace", "diffattn_v2_decode_workspace", "diffattn_decode_fp8k",
                 "diffattn_decode_noalloc", "diffattn_projection", "diffattn_forward_fp8qk", "diffattn_layer_forward",
                 "diffattn_v2_forward_fp8qk", "diffattn_bounds_checked", "diffattn_debug_bounds_selftest",
                 "diffattn_forward_train", "diffattn_backward_saved", "diffattn_forward_saved_bytes",
                 "diffattn_v2_forward_train", "diffattn_v2_backward_saved", "diffattn_v2_forward_saved_bytes",
                 "diffattn_layer_workspace", "diffattn_v2_layer_forward", "diffattn_v2_layer_workspace",
                 "diffattn_v2_decode_fp8k", "diffattn_backward", "diffattn_backward_workspace",
                 "lambda_reparam_backward", "diffattn_v2_backward", "diffattn_v2_backward_workspace"):
        assert want in names


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), f"{name} not exported"


def test_normal_build_has_no_bounds_checks(L):
    assert L.diffattn_bounds_checked() == 0
    assert L.diffattn_debug_bounds_selftest(None) == da.ERR_UNSUPPORTED  # refused on the host, nothing launched


def test_bounds_build_compiles_and_exports_the_same_symbols():
    path = build.build(bounds=True)
    assert path.endswith("libdiffattn_bounds.so")
    Lb = ctypes.CDLL(path)
    for name in _declared():
        assert hasattr(Lb, name), f"{name} not exported by the bounds-check build"
    Lb.diffattn_bounds_checked.restype = ctypes.c_int
    assert Lb.diffattn_bounds_checked() == 1


def test_lambda_init_host(L):
    for l in (1, 4, 12, 20):
        assert da.lambda_init(l) == pytest.approx(oracle.lambda_init(l), abs=1e-7)
    import math
    assert math.isnan(da.lambda_init(0))


P = ctypes.c_void_p
A = P(0x10000)        # 16-byte aligned fake device address (never dereferenced)
MIS = P(0x10008)      # misaligned fake address


def _fwd(L, dt=1, B=1, H=1, n=8, d=64, ptrs=None, lam=A, out=A):
    q = ptrs or [A] * 5
    return L.diffattn_forward(dt, B, H, n, d, *q, lam, ctypes.c_float(0.2), None, ctypes.c_float(1e-5), 1,
                              out, None)


def _v2(L, dt=1, B=1, Hq=4, Hkv=2, n=8, d=128, q=A, logits=A, sb=0, st=0):
    return L.diffattn_v2_forward(dt, B, Hq, Hkv, n, d, q, A, A, logits, sb, st, ctypes.c_float(0.0), 1, A, None)


def test_forward_host_validation(L):
    assert _fwd(L, dt=7) == da.ERR_DTYPE
    assert _fwd(L, n=-1) == da.ERR_SHAPE
    assert _fwd(L, d=0) == da.ERR_SHAPE
    assert _fwd(L, n=0) == da.OK           # empty input: no launch
    assert _fwd(L, B=0) == da.OK
    assert _fwd(L, ptrs=[A, None, A, A, A]) == da.ERR_NULL
    assert _fwd(L, lam=None) == da.ERR_NULL
    assert _fwd(L, out=None) == da.ERR_NULL
    assert _fwd(L, d=96) == da.ERR_UNSUPPORTED
    assert _fwd(L, dt=0, d=300) == da.ERR_UNSUPPORTED
    assert _fwd(L, ptrs=[A, A, MIS, A, A]) == da.ERR_ALIGN
    assert _fwd(L, out=MIS) == da.ERR_ALIGN
    assert b"16-byte" in L.diffattn_last_error()


def test_forward_host_workspace_size(L):
    def r256(x):
        return (x + 255) // 256 * 256
    for dt, es in ((1, 2), (0, 4)):
        for B, H, n, d in ((4, 16, 2048, 64), (1, 1, 1, 1), (3, 2, 129, 128)):
            qk = B * n * H * d * es
            assert L.diffattn_forward_host_workspace(dt, B, H, n, d) == 4 * r256(qk) + 2 * r256(2 * qk)
    assert L.diffattn_forward_host_workspace(7, 1, 1, 8, 64) == 0
    assert L.diffattn_forward_host_workspace(1, -1, 1, 8, 64) == 0


def test_forward_host_buffer_validation(L):
    """The host-buffer entry point rejects bad arguments before any CUDA call."""
    W = P(0x100000)  # 256-byte aligned fake device workspace (never dereferenced)
    need = L.diffattn_forward_host_workspace(1, 1, 1, 8, 64)

    def call(dt=1, B=1, n=8, d=64, q1=A, out=A, ws=W, nbytes=need):
        return L.diffattn_forward_host(dt, B, 1, n, d, q1, A, A, A, A, A, ctypes.c_float(0.2), None,
                                       ctypes.c_float(1e-5), 1, out, ws, nbytes, None)
    assert call(dt=7) == da.ERR_DTYPE
    assert call(n=-1) == da.ERR_SHAPE
    assert call(n=0) == da.OK
    assert call(q1=None) == da.ERR_NULL
    assert call(out=None) == da.ERR_NULL
    assert call(ws=None) == da.ERR_NULL
    assert call(nbytes=need - 1) == da.ERR_SHAPE
    assert b"workspace" in L.diffattn_last_error()
    assert call(ws=P(0x100010)) == da.ERR_ALIGN


def test_decode_host_validation(L):
    def call(dt=1, B=1, n=8, d=64, q1=A, out=A, k1=A):
        return L.diffattn_decode(dt, B, 2, n, d, q1, A, k1, A, A, None, A, ctypes.c_float(0.2), None,
                                 ctypes.c_float(1e-5), out, None, 0, None)
    assert call(dt=7) == da.ERR_DTYPE
    assert call(n=-1) == da.ERR_SHAPE
    assert call(B=0) == da.OK
    assert call(q1=None) == da.ERR_NULL
    assert call(out=None) == da.ERR_NULL
    assert call(dt=0) == da.ERR_UNSUPPORTED   # fp32 decode is not provided
    assert call(d=96) == da.ERR_UNSUPPORTED
    assert call(k1=MIS) == da.ERR_ALIGN


def test_decode_workspace_validation(L):
    """A workspace that is given must be large enough and 4-byte aligned (NULL is always fine)."""
    W = P(0x100000)
    need1 = L.diffattn_decode_workspace(1, 2, 64)
    need2 = L.diffattn_v2_decode_workspace(1, 4, 128)

    def v1(ws=W, nbytes=need1):
        return L.diffattn_decode(1, 1, 2, 8, 64, A, A, A, A, A, None, A, ctypes.c_float(0.2), None,
                                 ctypes.c_float(1e-5), A, ws, nbytes, None)

    def v2(ws=W, nbytes=need2):
        return L.diffattn_v2_decode(1, 1, 4, 2, 8, 128, A, A, A, None, A, 0, ctypes.c_float(0.0), A, ws, nbytes,
                                    None)

    def v1_fp8(ws=W, nbytes=need1):
        return L.diffattn_decode_fp8k(1, 2, 8, 64, A, A, A, A, ctypes.c_float(1.0), ctypes.c_float(1.0), A, None, A,
                                      ctypes.c_float(0.2), None, ctypes.c_float(1e-5), A, ws, nbytes, None)
    for call, need in ((v1, need1), (v2, need2), (v1_fp8, need1)):
        assert call(nbytes=need - 1) == da.ERR_SHAPE
        assert b"workspace" in L.diffattn_last_error()
        assert call(ws=P(0x100002)) == da.ERR_ALIGN


def test_decode_noalloc_host_validation(L):
    """The no-allocation decode rejects batches beyond its fixed scratch before any CUDA call."""
    def call(dt=1, B=1, H=2, n=8, d=64):
        return L.diffattn_decode_noalloc(dt, B, H, n, d, A, A, A, A, A, None, A, ctypes.c_float(0.2), None,
                                         ctypes.c_float(1e-5), A, None)
    assert call(B=255, H=1, d=128) == da.ERR_SHAPE      # 255 pairs x 16512 bytes > 4 MiB
    assert b"scratch" in L.diffattn_last_error()
    assert call(B=1, H=505, d=64) == da.ERR_SHAPE       # 505 pairs x 8320 bytes > 4 MiB
    assert call(B=0) == da.OK
    assert call(dt=7) == da.ERR_DTYPE
    assert call(dt=0) == da.ERR_UNSUPPORTED
    assert call(d=96) == da.ERR_UNSUPPORTED
    assert call(n=-1) == da.ERR_SHAPE


def test_decode_workspace_sizes(L):
    # Eight cluster states per (b, h) at most, each two maps x (maximum, sum, value-width channels), fp32.
    assert L.diffattn_decode_workspace(8, 16, 64) == 8 * 16 * 8 * 2 * (128 + 2) * 4
    assert L.diffattn_v2_decode_workspace(8, 32, 128) == 8 * 16 * 8 * 2 * (128 + 2) * 4
    assert L.diffattn_decode_workspace(-1, 16, 64) == 0


def test_v2_decode_host_validation(L):
    def call(dt=1, Hq=4, Hkv=2, n=8, d=128, q=A, sb=0):
        return L.diffattn_v2_decode(dt, 1, Hq, Hkv, n, d, q, A, A, None, A, sb, ctypes.c_float(0.0), A, None, 0,
                                    None)
    assert call(Hq=3, Hkv=1) == da.ERR_SHAPE
    assert call(Hq=6, Hkv=2) == da.ERR_SHAPE
    assert call(sb=-1) == da.ERR_SHAPE
    assert call(q=None) == da.ERR_NULL
    assert call(d=64) == da.ERR_UNSUPPORTED
    assert call(dt=0) == da.ERR_UNSUPPORTED
    assert call(q=MIS) == da.ERR_ALIGN


def test_fp8k_decode_host_validation(L):
    def v1(B=1, n=8, d=64, k1=A, s1=1.0, s2=1.0, out=A):
        return L.diffattn_decode_fp8k(B, 2, n, d, A, A, k1, A, ctypes.c_float(s1), ctypes.c_float(s2), A, None, A,
                                      ctypes.c_float(0.2), None, ctypes.c_float(1e-5), out, None, 0, None)
    assert v1(n=-1) == da.ERR_SHAPE
    assert v1(B=0) == da.OK
    assert v1(k1=None) == da.ERR_NULL
    assert v1(d=96) == da.ERR_UNSUPPORTED
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        assert v1(s1=bad) == da.ERR_SHAPE
        assert v1(s2=bad) == da.ERR_SHAPE
    assert b"scale" in L.diffattn_last_error()
    assert v1(k1=MIS) == da.ERR_ALIGN

    def v2(Hq=4, Hkv=2, d=128, k=A, s=1.0):
        return L.diffattn_v2_decode_fp8k(1, Hq, Hkv, 8, d, A, k, ctypes.c_float(s), A, None, A, 0,
                                         ctypes.c_float(0.0), A, None, 0, None)
    assert v2(Hq=6, Hkv=2) == da.ERR_SHAPE
    assert v2(k=None) == da.ERR_NULL
    assert v2(d=64) == da.ERR_UNSUPPORTED
    assert v2(s=0.0) == da.ERR_SHAPE
    assert v2(k=MIS) == da.ERR_ALIGN


def test_backward_host_validation(L):
    need = L.diffattn_backward_workspace(2, 3, 100, 64)
    R = 2 * 3 * 100
    ctas = 2 * 3 * 13  # 8-row blocks of the row pass
    r256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert need == r256(R * 128 * 4) + r256(6 * R * 4) + r256(ctas * 128 * 4)
    W = P(0x100000)

    def call(dt=0, B=2, n=100, d=64, q1=A, dlam=A, ws=W, nbytes=need):
        return L.diffattn_backward(dt, B, 3, n, d, q1, A, A, A, A, A, ctypes.c_float(0.2), None,
                                   ctypes.c_float(1e-5), 1, A, A, A, A, A, A, dlam, None, ws, nbytes, None)
    assert call(dt=7) == da.ERR_DTYPE
    assert call(dt=1, d=32) == da.ERR_UNSUPPORTED   # bf16 (tensor cores): d = 64 only
    assert call(dt=1, q1=MIS) == da.ERR_ALIGN       # bf16 tensors: 16-byte aligned
    assert call(d=129) == da.ERR_UNSUPPORTED
    assert call(n=-1) == da.ERR_SHAPE
    assert call(dlam=None) == da.ERR_NULL
    assert call(q1=None) == da.ERR_NULL
    assert call(ws=None) == da.ERR_NULL
    assert call(nbytes=need - 1) == da.ERR_SHAPE
    assert b"workspace" in L.diffattn_last_error()
    assert call(ws=P(0x100008)) == da.ERR_ALIGN
    assert L.lambda_reparam_backward(A, A, A, A, 8, None, A, A, A, A, None) == da.ERR_NULL
    assert L.lambda_reparam_backward(A, A, A, A, 0, A, A, A, A, A, None) == da.ERR_SHAPE


def test_v2_backward_host_validation(L):
    R = 2 * 2 * 50
    r256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    need = L.diffattn_v2_backward_workspace(2, 4, 50, 32)
    assert need == r256(R * 32 * 4) + r256(6 * R * 4)
    W = P(0x100000)

    def call(dt=0, Hq=4, Hkv=2, n=50, d=32, sb=0, st=0, q=A, dlog=A, ws=W, nbytes=need):
        return L.diffattn_v2_backward(dt, 2, Hq, Hkv, n, d, q, A, A, A, sb, st, ctypes.c_float(0.0), 1, A, A, A,
                                      A, dlog, ws, nbytes, None)
    assert call(dt=7) == da.ERR_DTYPE
    assert call(dt=1) == da.ERR_UNSUPPORTED
    assert call(Hq=6, Hkv=2) == da.ERR_SHAPE
    assert call(sb=-1) == da.ERR_SHAPE
    assert call(sb=3, st=0) == da.ERR_UNSUPPORTED        # neither per pair, per sequence nor per token
    assert call(sb=2, st=0, q=None) == da.ERR_NULL       # per sequence (Hq/2, 0): past the stride check
    assert call(sb=100, st=2, q=None) == da.ERR_NULL     # per token (n * Hq/2, Hq/2)
    assert call(dlog=None) == da.ERR_NULL
    assert call(nbytes=need - 1) == da.ERR_SHAPE
    assert call(ws=P(0x100008)) == da.ERR_ALIGN


def test_fp8qk_forward_host_validation(L):
    def call(B=1, H=2, n=8, d=128, q1=A, s=(1.0, 1.0, 1.0, 1.0), out=A):
        return L.diffattn_forward_fp8qk(B, H, n, d, q1, A, A, A, *(ctypes.c_float(x) for x in s), A, A,
                                        ctypes.c_float(0.2), None, ctypes.c_float(1e-5), 1, out, None)
    assert call(n=-1) == da.ERR_SHAPE
    assert call(d=96) == da.ERR_UNSUPPORTED
    assert call(d=64, H=1) == da.ERR_UNSUPPORTED  # d = 64 reads two heads' rows a box
    assert call(d=64, q1=None) == da.ERR_NULL
    assert call(d=64, B=0) == da.OK
    assert call(B=0) == da.OK
    assert call(q1=None) == da.ERR_NULL
    for bad in (0.0, -2.0, float("nan"), float("inf")):
        for i in range(4):
            sc = [1.0] * 4
            sc[i] = bad
            assert call(s=tuple(sc)) == da.ERR_SHAPE
    assert call(q1=MIS) == da.ERR_ALIGN
    assert call(out=MIS) == da.ERR_ALIGN


def test_v2_fp8qk_forward_host_validation(L):
    def call(B=1, Hq=4, Hkv=2, n=8, d=128, q=A, s=(1.0, 1.0), sb=0, st=0, out=A):
        return L.diffattn_v2_forward_fp8qk(B, Hq, Hkv, n, d, q, A, *(ctypes.c_float(x) for x in s), A, A, sb, st,
                                           ctypes.c_float(0.0), 1, out, None)
    assert call(n=-1) == da.ERR_SHAPE
    assert call(Hq=3) == da.ERR_SHAPE                # Hq odd
    assert call(Hq=4, Hkv=4) == da.ERR_SHAPE         # Hq / Hkv odd
    assert call(sb=-1) == da.ERR_SHAPE
    assert call(d=64) == da.ERR_UNSUPPORTED
    assert call(B=0) == da.OK
    assert call(q=None) == da.ERR_NULL
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        assert call(s=(bad, 1.0)) == da.ERR_SHAPE
        assert call(s=(1.0, bad)) == da.ERR_SHAPE
    assert call(q=MIS) == da.ERR_ALIGN
    assert call(out=MIS) == da.ERR_ALIGN


def test_training_pair_host_validation(L):
    sz = ctypes.c_size_t
    need = L.diffattn_forward_saved_bytes(1, 2, 8, 64)
    assert need >= 2 * 16 * 4 + 2 * 16 * 128 * 2
    SAVED = P(0x200000)  # 256-byte aligned fake device address

    def fwd(d=64, saved=SAVED, nbytes=None, q1=A):
        nb = need if nbytes is None else nbytes
        return L.diffattn_forward_train(1, 2, 8, d, q1, A, A, A, A, A, ctypes.c_float(0.2), None, ctypes.c_float(1e-5),
                                        1, A, saved, sz(nb), None)
    assert fwd(d=128) == da.ERR_UNSUPPORTED
    assert fwd(q1=None) == da.ERR_NULL
    assert fwd(saved=None) == da.ERR_NULL
    assert fwd(nbytes=need - 1) == da.ERR_SHAPE
    assert fwd(saved=P(0x200010)) == da.ERR_ALIGN
    assert fwd(q1=MIS) == da.ERR_ALIGN
    wneed = L.diffattn_backward_workspace(1, 2, 8, 64)

    def bwd(d=64, saved=SAVED, nbytes=None, ws=A, wbytes=None, dlam=A):
        nb = need if nbytes is None else nbytes
        wb = wneed if wbytes is None else wbytes
        return L.diffattn_backward_saved(1, 2, 8, d, A, A, A, A, A, A, ctypes.c_float(0.2), None,
                                         ctypes.c_float(1e-5), 1, A, saved, sz(nb), A, A, A, A, A, dlam, None, ws,
                                         sz(wb), None)
    assert bwd(d=128) == da.ERR_UNSUPPORTED
    assert bwd(dlam=None) == da.ERR_NULL
    assert bwd(saved=None) == da.ERR_NULL
    assert bwd(nbytes=need - 1) == da.ERR_SHAPE
    assert bwd(wbytes=wneed - 1) == da.ERR_SHAPE
    assert bwd(ws=MIS) == da.ERR_ALIGN
    need2 = L.diffattn_v2_forward_saved_bytes(1, 4, 8, 128)

    def fwd2(Hq=4, Hkv=2, d=128, saved=SAVED, nbytes=None, sb=0, st=0):
        nb = need2 if nbytes is None else nbytes
        return L.diffattn_v2_forward_train(1, Hq, Hkv, 8, d, A, A, A, A, sb, st, ctypes.c_float(0.0), 1, A, saved,
                                           sz(nb), None)
    assert fwd2(d=64) == da.ERR_UNSUPPORTED
    assert fwd2(Hq=3) == da.ERR_SHAPE
    assert fwd2(sb=-1) == da.ERR_SHAPE
    assert fwd2(saved=None) == da.ERR_NULL
    assert fwd2(nbytes=need2 - 1) == da.ERR_SHAPE
    w2 = L.diffattn_v2_backward_workspace(1, 4, 8, 128)

    def bwd2(d=128, sb=0, st=0, saved=SAVED, nbytes=None, wbytes=None):
        nb = need2 if nbytes is None else nbytes
        wb = w2 if wbytes is None else wbytes
        return L.diffattn_v2_backward_saved(1, 4, 2, 8, d, A, A, A, A, sb, st, ctypes.c_float(0.0), 1, A, saved,
                                            sz(nb), A, A, A, A, A, sz(wb), None)
    assert bwd2(d=64) == da.ERR_UNSUPPORTED
    assert bwd2(sb=3, st=1) == da.ERR_UNSUPPORTED  # not one of the three logit layouts
    assert bwd2(saved=None) == da.ERR_NULL
    assert bwd2(nbytes=need2 - 1) == da.ERR_SHAPE
    assert bwd2(wbytes=w2 - 1) == da.ERR_SHAPE


def test_projection_host_validation(L):
    def call(M=4, N=8, K=8, a=A, w=A, c=A):
        return L.diffattn_projection(M, N, K, a, w, c, None)
    assert call(M=-1) == da.ERR_SHAPE
    assert call(K=0) == da.ERR_SHAPE
    assert call(M=0) == da.OK and call(N=0) == da.OK
    assert call(a=None) == da.ERR_NULL
    assert call(K=12) == da.ERR_SHAPE      # rows must be 16-byte multiples
    assert call(N=12) == da.ERR_SHAPE
    assert call(w=MIS) == da.ERR_ALIGN


def test_layer_workspace_sizes(L):
    r256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    M, H, d = 2 * 100, 3, 64
    assert L.diffattn_layer_workspace(2, 100, H, d) == r256(M * 6 * H * d * 2) + r256(M * 2 * H * d * 2) + 256
    Hq, Hkv, d = 8, 2, 128
    nq = (Hq + 2 * Hkv) * d
    assert L.diffattn_v2_layer_workspace(2, 100, Hq, Hkv, d) == r256(M * nq * 2) + r256(M * 4 * 4) + r256(
        M * 4 * d * 2)
    assert L.diffattn_layer_workspace(-1, 100, H, 64) == 0


def test_layer_host_validation(L):
    W = P(0x100000)
    need = L.diffattn_layer_workspace(1, 8, 2, 64)

    def v1(B=1, n=8, D=256, H=2, d=64, x=A, lq=A, ws=W, nbytes=need):
        return L.diffattn_layer_forward(B, n, D, H, d, x, A, A, lq, A, A, A, ctypes.c_float(0.2), None,
                                        ctypes.c_float(1e-5), 1, A, ws, nbytes, None)
    assert v1(d=96) == da.ERR_UNSUPPORTED
    assert v1(D=250) == da.ERR_SHAPE
    assert v1(H=0) == da.ERR_SHAPE
    assert v1(B=0) == da.OK and v1(n=0) == da.OK
    assert v1(x=None) == da.ERR_NULL
    assert v1(lq=None) == da.ERR_NULL
    assert v1(x=MIS) == da.ERR_ALIGN
    assert v1(nbytes=need - 1) == da.ERR_SHAPE
    assert b"workspace" in L.diffattn_last_error()
    assert v1(ws=P(0x100010)) == da.ERR_ALIGN
    need2 = L.diffattn_v2_layer_workspace(1, 8, 4, 2, 128)

    def v2(Hq=4, Hkv=2, d=128, D=256, x=A, nbytes=need2):
        return L.diffattn_v2_layer_forward(1, 8, D, Hq, Hkv, d, x, A, A, 1, A, W, nbytes, None)
    assert v2(Hq=6, Hkv=2) == da.ERR_SHAPE
    assert v2(d=64) == da.ERR_UNSUPPORTED
    assert v2(D=100) == da.ERR_SHAPE
    assert v2(x=None) == da.ERR_NULL
    assert v2(nbytes=need2 - 1) == da.ERR_SHAPE


def test_v2_host_validation(L):
    assert _v2(L, Hq=3, Hkv=1) == da.ERR_SHAPE        # odd query heads
    assert _v2(L, Hq=6, Hkv=2) == da.ERR_SHAPE        # group of 3 would straddle a pair
    assert _v2(L, Hq=4, Hkv=3) == da.ERR_SHAPE
    assert _v2(L, Hkv=0) == da.ERR_SHAPE
    assert _v2(L, sb=-1) == da.ERR_SHAPE
    assert _v2(L, n=0) == da.OK
    assert _v2(L, q=None) == da.ERR_NULL
    assert _v2(L, logits=None) == da.ERR_NULL


def test_lambda_reparam_host_validation(L):
    assert L.lambda_reparam(A, A, A, None, 8, ctypes.c_float(0.2), A, None) == da.ERR_NULL
    assert L.lambda_reparam(A, A, A, A, 0, ctypes.c_float(0.2), A, None) == da.ERR_SHAPE


def test_debug_wait_budget_validation(L):
    assert L.diffattn_debug_wait_timeout(0, None) == da.ERR_SHAPE
    assert L.diffattn_debug_wait_timeout(2 * 10**9, None) == da.ERR_SHAPE


def test_product_path_has_no_fallback():
    """The binding never imports the oracle and raises if the library is missing."""
    src = open(os.path.join(ROOT, "differential_attention_03_gb300", "binding.py")).read()
    assert "oracle" not in src.replace("no fallback", "")
    for f in os.listdir(os.path.join(ROOT, "differential_attention_03_gb300")):
        if f.endswith(".py"):
            assert "import oracle" not in open(os.path.join(ROOT, "differential_attention_03_gb300", f)).read()
