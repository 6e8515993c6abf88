"""Thin ctypes binding over libdiffattn.so (argument marshalling only).

Every computation runs in the library's CUDA kernels; this module checks
tensor placement/dtype/contiguity, passes raw device pointers, sizes and the
current CUDA stream, and turns a non-OK status into an exception.  PyTorch is
used only for device memory and streams.  If the library is missing this
module raises on first use: there is no fallback path.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# DIFFATTN_DEBUG=1 loads the bounds-check build (every TMA coordinate, TMEM
# address and global store of the kernels checked; see build.py) instead.
BOUNDS = os.environ.get("DIFFATTN_DEBUG", "") == "1"
LIB_PATH = os.path.join(_PKG, "libdiffattn_bounds.so" if BOUNDS else "libdiffattn.so")

OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_DTYPE, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_BOUNDS = range(9)
STATUS_NAMES = ["OK", "ERR_NULL", "ERR_SHAPE", "ERR_ALIGN", "ERR_DTYPE", "ERR_UNSUPPORTED", "ERR_CUDA",
                "ERR_TIMEOUT", "ERR_BOUNDS"]
F32, BF16 = 0, 1

_lock = threading.Lock()
_lib = None


class DiffAttnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        self.status = status
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{name}: {msg}")


def lib() -> ctypes.CDLL:
    """Load libdiffattn.so (built in-tree by ``build.py``); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -m differential_attention_03_gb300.build`"
                                   + (" --bounds" if BOUNDS else ""))
            L = ctypes.CDLL(LIB_PATH)
            vp, i, f, ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_longlong
            L.diffattn_lambda_init.argtypes = [i]
            L.diffattn_lambda_init.restype = f
            L.lambda_reparam.argtypes = [vp, vp, vp, vp, i, f, vp, vp]
            L.lambda_reparam.restype = i
            L.diffattn_forward.argtypes = [i, i, i, i, i, vp, vp, vp, vp, vp, vp, f, vp, f, i, vp, vp]
            L.diffattn_forward.restype = i
            L.diffattn_forward_host_workspace.argtypes = [i, i, i, i, i]
            L.diffattn_forward_host_workspace.restype = ctypes.c_size_t
            L.diffattn_forward_host.argtypes = [i, i, i, i, i, vp, vp, vp, vp, vp, vp, f, vp, f, i, vp, vp,
                                                ctypes.c_size_t, vp]
            L.diffattn_forward_host.restype = i
            L.diffattn_decode_workspace.argtypes = [i, i, i]
            L.diffattn_decode_workspace.restype = ctypes.c_size_t
            L.diffattn_v2_decode_workspace.argtypes = [i, i, i]
            L.diffattn_v2_decode_workspace.restype = ctypes.c_size_t
            L.diffattn_decode.argtypes = [i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp, f, vp, f, vp, vp,
                                          ctypes.c_size_t, vp]
            L.diffattn_decode.restype = i
            L.diffattn_decode_noalloc.argtypes = [i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp, f, vp, f, vp, vp]
            L.diffattn_decode_noalloc.restype = i
            L.diffattn_v2_decode.argtypes = [i, i, i, i, i, i, vp, vp, vp, vp, vp, ll, f, vp, vp, ctypes.c_size_t,
                                             vp]
            L.diffattn_v2_decode.restype = i
            L.diffattn_decode_fp8k.argtypes = [i, i, i, i, vp, vp, vp, vp, f, f, vp, vp, vp, f, vp, f, vp, vp,
                                               ctypes.c_size_t, vp]
            L.diffattn_decode_fp8k.restype = i
            L.diffattn_v2_decode_fp8k.argtypes = [i, i, i, i, i, vp, vp, f, vp, vp, vp, ll, f, vp, vp,
                                                  ctypes.c_size_t, vp]
            L.diffattn_v2_decode_fp8k.restype = i
            L.diffattn_backward_workspace.argtypes = [i, i, i, i]
            L.diffattn_backward_workspace.restype = ctypes.c_size_t
            L.diffattn_backward.argtypes = [i, i, i, i, i, vp, vp, vp, vp, vp, vp, f, vp, f, i, vp, vp, vp, vp, vp,
                                            vp, vp, vp, vp, ctypes.c_size_t, vp]
            L.diffattn_backward.restype = i
            L.diffattn_v2_backward_workspace.argtypes = [i, i, i, i]
            L.diffattn_v2_backward_workspace.restype = ctypes.c_size_t
            L.diffattn_v2_backward.argtypes = [i, i, i, i, i, i, vp, vp, vp, vp, ll, ll, f, i, vp, vp, vp, vp, vp,
                                               vp, ctypes.c_size_t, vp]
            L.diffattn_v2_backward.restype = i
            L.lambda_reparam_backward.argtypes = [vp, vp, vp, vp, i, vp, vp, vp, vp, vp, vp]
            L.lambda_reparam_backward.restype = i
            L.diffattn_v2_forward.argtypes = [i, i, i, i, i, i, vp, vp, vp, vp, ll, ll, f, i, vp, vp]
            L.diffattn_v2_forward.restype = i
            L.diffattn_forward_fp8qk.argtypes = [i, i, i, i, vp, vp, vp, vp, f, f, f, f, vp, vp, f, vp, f, i, vp, vp]
            L.diffattn_forward_fp8qk.restype = i
            L.diffattn_v2_forward_fp8qk.argtypes = [i, i, i, i, i, vp, vp, f, f, vp, vp, ll, ll, f, i, vp, vp]
            L.diffattn_v2_forward_fp8qk.restype = i
            sz = ctypes.c_size_t
            L.diffattn_forward_saved_bytes.argtypes = [i, i, i, i]
            L.diffattn_forward_saved_bytes.restype = sz
            L.diffattn_v2_forward_saved_bytes.argtypes = [i, i, i, i]
            L.diffattn_v2_forward_saved_bytes.restype = sz
            L.diffattn_forward_train.argtypes = [i, i, i, i, vp, vp, vp, vp, vp, vp, f, vp, f, i, vp, vp, sz, vp]
            L.diffattn_forward_train.restype = i
            L.diffattn_backward_saved.argtypes = [i, i, i, i, vp, vp, vp, vp, vp, vp, f, vp, f, i, vp, vp, sz,
                                                  vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
            L.diffattn_backward_saved.restype = i
            L.diffattn_v2_forward_train.argtypes = [i, i, i, i, i, vp, vp, vp, vp, ll, ll, f, i, vp, vp, sz, vp]
            L.diffattn_v2_forward_train.restype = i
            L.diffattn_v2_backward_saved.argtypes = [i, i, i, i, i, vp, vp, vp, vp, ll, ll, f, i, vp, vp, sz,
                                                     vp, vp, vp, vp, vp, sz, vp]
            L.diffattn_v2_backward_saved.restype = i
            L.diffattn_projection.argtypes = [i, i, i, vp, vp, vp, vp]
            L.diffattn_projection.restype = i
            L.diffattn_layer_workspace.argtypes = [i, i, i, i]
            L.diffattn_layer_workspace.restype = ctypes.c_size_t
            L.diffattn_layer_forward.argtypes = [i, i, i, i, i, vp, vp, vp, vp, vp, vp, vp, f, vp, f, i, vp, vp,
                                                 ctypes.c_size_t, vp]
            L.diffattn_layer_forward.restype = i
            L.diffattn_v2_layer_workspace.argtypes = [i, i, i, i, i]
            L.diffattn_v2_layer_workspace.restype = ctypes.c_size_t
            L.diffattn_v2_layer_forward.argtypes = [i, i, i, i, i, i, vp, vp, vp, i, vp, vp, ctypes.c_size_t, vp]
            L.diffattn_v2_layer_forward.restype = i
            L.diffattn_device_status.argtypes = [vp]
            L.diffattn_device_status.restype = i
            L.diffattn_bounds_checked.argtypes = []
            L.diffattn_bounds_checked.restype = i
            L.diffattn_debug_bounds_selftest.argtypes = [vp]
            L.diffattn_debug_bounds_selftest.restype = i
            L.diffattn_debug_item_plan.argtypes = [i, ll, i, i, i, i, ll, vp, vp]
            L.diffattn_debug_item_plan.restype = i
            L.diffattn_last_error.argtypes = []
            L.diffattn_last_error.restype = ctypes.c_char_p
            L.diffattn_debug_wait_timeout.argtypes = [ll, vp]
            L.diffattn_debug_wait_timeout.restype = i
            L.diffattn_launch_count.argtypes = []
            L.diffattn_launch_count.restype = ll
            _lib = L
    return _lib


def _check(status: int):
    if status != OK:
        raise DiffAttnError(status, lib().diffattn_last_error().decode(errors="replace"))


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise ValueError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def lambda_init(layer_index: int) -> float:
    """lambda_init = 0.8 - 0.6 exp(-0.3 (l - 1)) for the 1-based layer index (host)."""
    return float(lib().diffattn_lambda_init(int(layer_index)))


def lambda_reparam(lq1, lk1, lq2, lk2, lambda_init_value: float, out=None, stream=None) -> torch.Tensor:
    """Device scalar lambda = exp(lq1.lk1) - exp(lq2.lk2) + lambda_init (fp32, one element)."""
    for name, t in (("lq1", lq1), ("lk1", lk1), ("lq2", lq2), ("lk2", lk2)):
        _need(t, name, torch.float32, (lq1.numel(),))
    if out is None:
        out = torch.empty(1, device=lq1.device, dtype=torch.float32)
    _need(out, "out", torch.float32, (1,))
    _check(lib().lambda_reparam(_ptr(lq1), _ptr(lk1), _ptr(lq2), _ptr(lk2), lq1.numel(),
                                float(lambda_init_value), _ptr(out), _stream(stream)))
    return out


def diffattn_forward(q1, q2, k1, k2, v, lam, lambda_init_value: float, gamma=None, eps: float = 1e-5,
                     causal: bool = True, out=None, stream=None) -> torch.Tensor:
    """DIFF V1 forward with per-head RMSNorm x (1 - lambda_init); BSHD tensors.

    q1, q2, k1, k2: [B, n, H, d]; v: [B, n, H, 2d]; lam: device fp32 scalar
    tensor; gamma: fp32 [2d] or None.  Returns out [B, n, H, 2d] (input dtype).
    """
    B, n, H, d = q1.shape
    dt = q1.dtype
    for name, t in (("q1", q1), ("q2", q2), ("k1", k1), ("k2", k2)):
        _need(t, name, dt, (B, n, H, d))
    _need(v, "v", dt, (B, n, H, 2 * d))
    _need(lam, "lambda", torch.float32, (1,))
    if gamma is not None:
        _need(gamma, "gamma", torch.float32, (2 * d,))
    if out is None:
        out = torch.empty((B, n, H, 2 * d), device=q1.device, dtype=dt)
    _need(out, "out", dt, (B, n, H, 2 * d))
    _check(lib().diffattn_forward(_dt(q1), B, H, n, d, _ptr(q1), _ptr(q2), _ptr(k1), _ptr(k2), _ptr(v),
                                  _ptr(lam), float(lambda_init_value), _ptr(gamma), float(eps),
                                  1 if causal else 0, _ptr(out), _stream(stream)))
    return out


def diffattn_forward_fp8qk(q1, q2, k1, k2, scales, v, lam, lambda_init_value: float, gamma=None, eps: float = 1e-5,
                           causal: bool = True, out=None, stream=None) -> torch.Tensor:
    """DIFF V1 forward with e4m3 queries and keys (QK^T on the FP8 tensor-core path).

    q1, q2, k1, k2: [B, n, H, d] e4m3 codes (torch.float8_e4m3fn or their bytes as uint8) of
    Q_r / q_scale_r and K_r / k_scale_r, d = 128, or d = 64 with H >= 2; scales = (q1_scale,
    q2_scale, k1_scale, k2_scale).  The result is diffattn_forward's for Q_r = q_scale_r e4m3(q_r),
    K_r = k_scale_r e4m3(k_r); v bf16 [B, n, H, 2d].  Returns out [B, n, H, 2d] bf16.
    """
    B, n, H, d = q1.shape
    for name, t in (("q1", q1), ("q2", q2), ("k1", k1), ("k2", k2)):
        _need_fp8(t, name, (B, n, H, d))
    _need(v, "v", torch.bfloat16, (B, n, H, 2 * d))
    _need(lam, "lambda", torch.float32, (1,))
    if gamma is not None:
        _need(gamma, "gamma", torch.float32, (2 * d,))
    if out is None:
        out = torch.empty((B, n, H, 2 * d), device=v.device, dtype=torch.bfloat16)
    _need(out, "out", torch.bfloat16, (B, n, H, 2 * d))
    s1, s2, s3, s4 = (float(x) for x in scales)
    _check(lib().diffattn_forward_fp8qk(B, H, n, d, _ptr(q1), _ptr(q2), _ptr(k1), _ptr(k2), s1, s2, s3, s4, _ptr(v),
                                        _ptr(lam), float(lambda_init_value), _ptr(gamma), float(eps),
                                        1 if causal else 0, _ptr(out), _stream(stream)))
    return out


def _need_host(t: torch.Tensor, name: str, dtype=None, shape=None):
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def forward_host_workspace_bytes(dtype, B: int, H: int, n: int, d: int) -> int:
    """Device workspace (bytes) that diffattn_forward_host needs for these sizes."""
    return int(lib().diffattn_forward_host_workspace(BF16 if dtype == torch.bfloat16 else F32, B, H, n, d))


def diffattn_forward_host(q1, q2, k1, k2, v, lam, lambda_init_value: float, gamma=None, eps: float = 1e-5,
                          causal: bool = True, out=None, workspace=None, stream=None) -> torch.Tensor:
    """diffattn_forward on HOST tensors (page-locked for asynchronous copies).

    The library copies the inputs in, runs the forward and copies the output
    back, pipelined over chunks of the batch.  lam / gamma are device tensors
    (layer parameters); workspace is a device uint8 tensor of at least
    forward_host_workspace_bytes(...) bytes (allocated here if None).  The host
    output is complete once `stream` (default: the current stream) has
    reached this call.
    """
    B, n, H, d = q1.shape
    dt = q1.dtype
    for name, t in (("q1", q1), ("q2", q2), ("k1", k1), ("k2", k2)):
        _need_host(t, name, dt, (B, n, H, d))
    _need_host(v, "v", dt, (B, n, H, 2 * d))
    _need(lam, "lambda", torch.float32, (1,))
    if gamma is not None:
        _need(gamma, "gamma", torch.float32, (2 * d,))
    if out is None:
        out = torch.empty((B, n, H, 2 * d), dtype=dt).pin_memory()
    _need_host(out, "out", dt, (B, n, H, 2 * d))
    need = forward_host_workspace_bytes(dt, B, H, n, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=lam.device)
    if not workspace.is_cuda or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace must be a CUDA tensor of at least {need} bytes")
    _check(lib().diffattn_forward_host(_dt(q1), B, H, n, d, _ptr(q1), _ptr(q2), _ptr(k1), _ptr(k2), _ptr(v),
                                       _ptr(lam), float(lambda_init_value), _ptr(gamma), float(eps),
                                       1 if causal else 0, _ptr(out), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def _ws_args(workspace, need):
    if workspace is None:
        return None, 0
    nbytes = workspace.numel() * workspace.element_size()
    if not workspace.is_cuda or nbytes < need:
        raise ValueError(f"workspace must be a CUDA tensor of at least {need} bytes")
    return _ptr(workspace), nbytes


def decode_workspace_bytes(B: int, H: int, d: int) -> int:
    """Device workspace that lets diffattn_decode split a (b, h) pair over several clusters."""
    return int(lib().diffattn_decode_workspace(B, H, d))


def v2_decode_workspace_bytes(B: int, Hq: int, d: int) -> int:
    return int(lib().diffattn_v2_decode_workspace(B, Hq, d))


def diffattn_decode(q1, q2, k1, k2, v, lam, lambda_init_value: float, gamma=None, eps: float = 1e-5,
                    lens=None, out=None, workspace=None, stream=None) -> torch.Tensor:
    """DIFF V1 decode: one new token per sequence over a key/value cache.

    q1, q2: [B, H, d]; k1, k2: [B, n, H, d]; v: [B, n, H, 2d] (bf16, d in
    {64, 128}); lens: int32 [B] visible keys per sequence or None (all n).
    workspace: None or a device tensor of decode_workspace_bytes(B, H, d)
    bytes (lets few (b, h) pairs use the whole GPU).  Returns out [B, H, 2d].
    """
    B, n, H, d = k1.shape
    dt = k1.dtype
    _need(q1, "q1", dt, (B, H, d))
    _need(q2, "q2", dt, (B, H, d))
    _need(k1, "k1", dt, (B, n, H, d))
    _need(k2, "k2", dt, (B, n, H, d))
    _need(v, "v", dt, (B, n, H, 2 * d))
    _need(lam, "lambda", torch.float32, (1,))
    if gamma is not None:
        _need(gamma, "gamma", torch.float32, (2 * d,))
    if lens is not None:
        _need(lens, "lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, H, 2 * d), device=k1.device, dtype=dt)
    _need(out, "out", dt, (B, H, 2 * d))
    wp, wn = _ws_args(workspace, decode_workspace_bytes(B, H, d))
    _check(lib().diffattn_decode(_dt(k1), B, H, n, d, _ptr(q1), _ptr(q2), _ptr(k1), _ptr(k2), _ptr(v),
                                 _ptr(lens), _ptr(lam), float(lambda_init_value), _ptr(gamma), float(eps),
                                 _ptr(out), wp, wn, _stream(stream)))
    return out


def diffattn_decode_noalloc(q1, q2, k1, k2, v, lam, lambda_init_value: float, gamma=None, eps: float = 1e-5,
                            lens=None, out=None, stream=None) -> torch.Tensor:
    """diffattn_decode for callers that cannot allocate device memory.

    Same arguments and result as diffattn_decode with a workspace, but the
    split states live in a fixed 4 MiB scratch inside the library (B*H at
    most 504 pairs at d = 64, 254 at d = 128).  Calls that can overlap on the
    GPU share that scratch and must be serialised on one stream.  ``out`` is
    allocated here with torch when None; pass it to allocate nothing.
    """
    B, n, H, d = k1.shape
    dt = k1.dtype
    _need(q1, "q1", dt, (B, H, d))
    _need(q2, "q2", dt, (B, H, d))
    _need(k1, "k1", dt, (B, n, H, d))
    _need(k2, "k2", dt, (B, n, H, d))
    _need(v, "v", dt, (B, n, H, 2 * d))
    _need(lam, "lambda", torch.float32, (1,))
    if gamma is not None:
        _need(gamma, "gamma", torch.float32, (2 * d,))
    if lens is not None:
        _need(lens, "lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, H, 2 * d), device=k1.device, dtype=dt)
    _need(out, "out", dt, (B, H, 2 * d))
    _check(lib().diffattn_decode_noalloc(_dt(k1), B, H, n, d, _ptr(q1), _ptr(q2), _ptr(k1), _ptr(k2), _ptr(v),
                                         _ptr(lens), _ptr(lam), float(lambda_init_value), _ptr(gamma), float(eps),
                                         _ptr(out), _stream(stream)))
    return out


def diffattn_v2_decode(q, k, v, lam_logits, lens=None, softmax_scale: float = 0.0, out=None,
                       workspace=None, stream=None) -> torch.Tensor:
    """DIFF V2 decode: one new token per sequence over a key/value cache.

    q: [B, Hq, d]; k, v: [B, n, Hkv, d] (bf16, d = 128); lam_logits: fp32
    [B, Hq/2] (one logit per pair of each sequence) or [Hq/2] (shared by all
    sequences); lens: int32 [B] or None.  Returns out [B, Hq/2, d].
    """
    B, n, Hkv, d = k.shape
    Hq = q.shape[1]
    dt = k.dtype
    _need(q, "q", dt, (B, Hq, d))
    _need(k, "k", dt, (B, n, Hkv, d))
    _need(v, "v", dt, (B, n, Hkv, d))
    if lam_logits.dim() == 1:
        _need(lam_logits, "lam_logits", torch.float32, (Hq // 2,))
        sb = 0
    else:
        _need(lam_logits, "lam_logits", torch.float32, (B, Hq // 2))
        sb = Hq // 2
    if lens is not None:
        _need(lens, "lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, Hq // 2, d), device=k.device, dtype=dt)
    _need(out, "out", dt, (B, Hq // 2, d))
    wp, wn = _ws_args(workspace, v2_decode_workspace_bytes(B, Hq, d))
    _check(lib().diffattn_v2_decode(_dt(k), B, Hq, Hkv, n, d, _ptr(q), _ptr(k), _ptr(v), _ptr(lens),
                                    _ptr(lam_logits), sb, float(softmax_scale), _ptr(out), wp, wn,
                                    _stream(stream)))
    return out


def _need_fp8(t: torch.Tensor, name: str, shape):
    if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise ValueError(f"{name} must hold e4m3 bytes (torch.float8_e4m3fn or torch.uint8), got {t.dtype}")
    _need(t, name, None, shape)


def diffattn_decode_fp8k(q1, q2, k1, k2, k1_scale: float, k2_scale: float, v, lam, lambda_init_value: float,
                         gamma=None, eps: float = 1e-5, lens=None, out=None, workspace=None,
                         stream=None) -> torch.Tensor:
    """DIFF V1 decode over an FP8 key cache.

    k1, k2: [B, n, H, d] e4m3 codes (torch.float8_e4m3fn or their bytes as
    torch.uint8) of K_r / k_scale_r; the result is diffattn_decode's for the
    keys k_scale_r * k_r.  q1, q2, v, lam, gamma, lens, workspace: as for
    diffattn_decode (bf16, d in {64, 128}).  Returns out [B, H, 2d] (bf16).
    """
    B, n, H, d = k1.shape
    _need(q1, "q1", torch.bfloat16, (B, H, d))
    _need(q2, "q2", torch.bfloat16, (B, H, d))
    _need_fp8(k1, "k1", (B, n, H, d))
    _need_fp8(k2, "k2", (B, n, H, d))
    _need(v, "v", torch.bfloat16, (B, n, H, 2 * d))
    _need(lam, "lambda", torch.float32, (1,))
    if gamma is not None:
        _need(gamma, "gamma", torch.float32, (2 * d,))
    if lens is not None:
        _need(lens, "lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, H, 2 * d), device=v.device, dtype=torch.bfloat16)
    _need(out, "out", torch.bfloat16, (B, H, 2 * d))
    wp, wn = _ws_args(workspace, decode_workspace_bytes(B, H, d))
    _check(lib().diffattn_decode_fp8k(B, H, n, d, _ptr(q1), _ptr(q2), _ptr(k1), _ptr(k2), float(k1_scale),
                                      float(k2_scale), _ptr(v), _ptr(lens), _ptr(lam), float(lambda_init_value),
                                      _ptr(gamma), float(eps), _ptr(out), wp, wn, _stream(stream)))
    return out


def diffattn_v2_decode_fp8k(q, k, k_scale: float, v, lam_logits, lens=None, softmax_scale: float = 0.0,
                            out=None, workspace=None, stream=None) -> torch.Tensor:
    """DIFF V2 decode over an FP8 key cache.

    k: [B, n, Hkv, d] e4m3 codes of K / k_scale (torch.float8_e4m3fn or
    torch.uint8); everything else as for diffattn_v2_decode (bf16, d = 128).
    Returns out [B, Hq/2, d] (bf16).
    """
    B, n, Hkv, d = k.shape
    Hq = q.shape[1]
    _need(q, "q", torch.bfloat16, (B, Hq, d))
    _need_fp8(k, "k", (B, n, Hkv, d))
    _need(v, "v", torch.bfloat16, (B, n, Hkv, d))
    if lam_logits.dim() == 1:
        _need(lam_logits, "lam_logits", torch.float32, (Hq // 2,))
        sb = 0
    else:
        _need(lam_logits, "lam_logits", torch.float32, (B, Hq // 2))
        sb = Hq // 2
    if lens is not None:
        _need(lens, "lens", torch.int32, (B,))
    if out is None:
        out = torch.empty((B, Hq // 2, d), device=v.device, dtype=torch.bfloat16)
    _need(out, "out", torch.bfloat16, (B, Hq // 2, d))
    wp, wn = _ws_args(workspace, v2_decode_workspace_bytes(B, Hq, d))
    _check(lib().diffattn_v2_decode_fp8k(B, Hq, Hkv, n, d, _ptr(q), _ptr(k), float(k_scale), _ptr(v), _ptr(lens),
                                         _ptr(lam_logits), sb, float(softmax_scale), _ptr(out), wp, wn,
                                         _stream(stream)))
    return out


def backward_workspace_bytes(B: int, H: int, n: int, d: int) -> int:
    """Device workspace diffattn_backward needs (per-row statistics, dO, dgamma shares)."""
    return int(lib().diffattn_backward_workspace(B, H, n, d))


def diffattn_backward(q1, q2, k1, k2, v, lam, lambda_init_value: float, dy, gamma=None, eps: float = 1e-5,
                      causal: bool = True, workspace=None, stream=None) -> dict:
    """DIFF V1 backward: gradients of diffattn_forward's output given dy.

    Shapes as for diffattn_forward; fp32 inputs (d <= 128, CUDA cores) or bf16
    inputs (d = 64, tensor cores); dy: [B, n, H, 2d] in the inputs' dtype.
    Returns a dict of fp32 gradients: dq1, dq2, dk1, dk2, dv (shaped like
    their inputs), dlam [1], dgamma [2d].  workspace: None (allocated here
    with torch) or a device tensor of backward_workspace_bytes(B, H, n, d) bytes.
    """
    B, n, H, d = q1.shape
    dt = q1.dtype
    for name, t, shp in (("q1", q1, (B, n, H, d)), ("q2", q2, (B, n, H, d)), ("k1", k1, (B, n, H, d)),
                         ("k2", k2, (B, n, H, d)), ("v", v, (B, n, H, 2 * d)), ("dy", dy, (B, n, H, 2 * d))):
        _need(t, name, dt, shp)
    _need(lam, "lambda", torch.float32, (1,))
    if gamma is not None:
        _need(gamma, "gamma", torch.float32, (2 * d,))
    need = backward_workspace_bytes(B, H, n, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q1.device)
    wp, wn = _ws_args(workspace, need)
    g = {k: torch.empty(t.shape, device=t.device, dtype=torch.float32)
         for k, t in (("dq1", q1), ("dq2", q2), ("dk1", k1), ("dk2", k2), ("dv", v))}
    g["dlam"] = torch.empty(1, device=q1.device, dtype=torch.float32)
    g["dgamma"] = torch.empty(2 * d, device=q1.device, dtype=torch.float32)
    _check(lib().diffattn_backward(_dt(q1), B, H, n, d, _ptr(q1), _ptr(q2), _ptr(k1), _ptr(k2), _ptr(v), _ptr(lam),
                                   float(lambda_init_value), _ptr(gamma), float(eps), 1 if causal else 0, _ptr(dy),
                                   _ptr(g["dq1"]), _ptr(g["dq2"]), _ptr(g["dk1"]), _ptr(g["dk2"]), _ptr(g["dv"]),
                                   _ptr(g["dlam"]), _ptr(g["dgamma"]), wp, wn, _stream(stream)))
    return g


def v2_backward_workspace_bytes(B: int, Hq: int, n: int, d: int) -> int:
    return int(lib().diffattn_v2_backward_workspace(B, Hq, n, d))


def diffattn_v2_backward(q, k, v, lam_logits, dy, causal: bool = True, softmax_scale: float = 0.0,
                         workspace=None, stream=None) -> dict:
    """DIFF V2 backward: gradients of diffattn_v2_forward's output given dy.

    q: [B, n, Hq, d]; k, v: [B, n, Hkv, d]; dy: [B, n, Hq/2, d], all fp32
    (d <= 128, CUDA cores) or all bf16 (d = 128, tensor cores); lam_logits:
    fp32 [B, n, Hq/2] (per token), [B, Hq/2] (per sequence) or [Hq/2] (per
    pair).  Returns a dict of fp32 gradients: dq, dk, dv and dlogits (shaped
    like lam_logits).
    """
    B, n, Hq, d = q.shape
    Hkv = k.shape[2]
    dt = q.dtype
    _need(q, "q", dt, (B, n, Hq, d))
    _need(k, "k", dt, (B, n, Hkv, d))
    _need(v, "v", dt, (B, n, Hkv, d))
    _need(dy, "dy", dt, (B, n, Hq // 2, d))
    G = Hq // 2
    f32 = torch.float32
    if lam_logits.dim() == 3:
        _need(lam_logits, "lam_logits", f32, (B, n, G))
        sb, st = n * G, G
    elif lam_logits.dim() == 2:
        _need(lam_logits, "lam_logits", f32, (B, G))
        sb, st = G, 0
    else:
        _need(lam_logits, "lam_logits", f32, (G,))
        sb, st = 0, 0
    need = v2_backward_workspace_bytes(B, Hq, n, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    wp, wn = _ws_args(workspace, need)
    g = {"dq": torch.empty(q.shape, device=q.device, dtype=f32), "dk": torch.empty(k.shape, device=q.device, dtype=f32),
         "dv": torch.empty(v.shape, device=q.device, dtype=f32), "dlogits": torch.empty_like(lam_logits)}
    _check(lib().diffattn_v2_backward(_dt(q), B, Hq, Hkv, n, d, _ptr(q), _ptr(k), _ptr(v), _ptr(lam_logits), sb, st,
                                      float(softmax_scale), 1 if causal else 0, _ptr(dy), _ptr(g["dq"]),
                                      _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["dlogits"]), wp, wn, _stream(stream)))
    return g


# ----------------------------------------------------------------------------- training pair
def forward_saved_bytes(B: int, H: int, n: int, d: int) -> int:
    """Device bytes that diffattn_forward_train saves for the backward (V1)."""
    return int(lib().diffattn_forward_saved_bytes(B, H, n, d))


def v2_forward_saved_bytes(B: int, Hq: int, n: int, d: int) -> int:
    """Device bytes that diffattn_v2_forward_train saves for the backward (V2)."""
    return int(lib().diffattn_v2_forward_saved_bytes(B, Hq, n, d))


def _saved_buf(saved, need, device):
    if saved is None:
        saved = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    if not saved.is_cuda or saved.dtype != torch.uint8 or saved.numel() < need:
        raise ValueError(f"saved must be a device uint8 tensor of at least {need} bytes")
    return saved


def diffattn_forward_train(q1, q2, k1, k2, v, lam, lambda_init_value: float, gamma=None, eps: float = 1e-5,
                           causal: bool = True, out=None, saved=None, stream=None):
    """diffattn_forward (bf16, d = 64) that also saves each row's lse and O_1, O_2 for
    diffattn_backward_saved.  Returns (out, saved)."""
    B, n, H, d = q1.shape
    for name, t, shp in (("q1", q1, (B, n, H, d)), ("q2", q2, (B, n, H, d)), ("k1", k1, (B, n, H, d)),
                         ("k2", k2, (B, n, H, d)), ("v", v, (B, n, H, 2 * d))):
        _need(t, name, torch.bfloat16, shp)
    _need(lam, "lambda", torch.float32, (1,))
    if gamma is not None:
        _need(gamma, "gamma", torch.float32, (2 * d,))
    if out is None:
        out = torch.empty((B, n, H, 2 * d), device=q1.device, dtype=torch.bfloat16)
    _need(out, "out", torch.bfloat16, (B, n, H, 2 * d))
    need = forward_saved_bytes(B, H, n, d)
    saved = _saved_buf(saved, need, q1.device)
    _check(lib().diffattn_forward_train(B, H, n, d, _ptr(q1), _ptr(q2), _ptr(k1), _ptr(k2), _ptr(v), _ptr(lam),
                                        float(lambda_init_value), _ptr(gamma), float(eps), 1 if causal else 0,
                                        _ptr(out), _ptr(saved), saved.numel(), _stream(stream)))
    return out, saved


def diffattn_backward_saved(q1, q2, k1, k2, v, lam, lambda_init_value: float, dy, saved, gamma=None,
                            eps: float = 1e-5, causal: bool = True, workspace=None, stream=None) -> dict:
    """diffattn_backward (bf16, d = 64) from the `saved` of diffattn_forward_train on the same inputs."""
    B, n, H, d = q1.shape
    for name, t, shp in (("q1", q1, (B, n, H, d)), ("q2", q2, (B, n, H, d)), ("k1", k1, (B, n, H, d)),
                         ("k2", k2, (B, n, H, d)), ("v", v, (B, n, H, 2 * d)), ("dy", dy, (B, n, H, 2 * d))):
        _need(t, name, torch.bfloat16, shp)
    _need(lam, "lambda", torch.float32, (1,))
    if gamma is not None:
        _need(gamma, "gamma", torch.float32, (2 * d,))
    need = backward_workspace_bytes(B, H, n, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q1.device)
    wp, wn = _ws_args(workspace, need)
    g = {k: torch.empty(t.shape, device=t.device, dtype=torch.float32)
         for k, t in (("dq1", q1), ("dq2", q2), ("dk1", k1), ("dk2", k2), ("dv", v))}
    g["dlam"] = torch.empty(1, device=q1.device, dtype=torch.float32)
    g["dgamma"] = torch.empty(2 * d, device=q1.device, dtype=torch.float32)
    _check(lib().diffattn_backward_saved(B, H, n, d, _ptr(q1), _ptr(q2), _ptr(k1), _ptr(k2), _ptr(v), _ptr(lam),
                                         float(lambda_init_value), _ptr(gamma), float(eps), 1 if causal else 0,
                                         _ptr(dy), _ptr(saved), saved.numel(), _ptr(g["dq1"]), _ptr(g["dq2"]),
                                         _ptr(g["dk1"]), _ptr(g["dk2"]), _ptr(g["dv"]), _ptr(g["dlam"]),
                                         _ptr(g["dgamma"]), wp, wn, _stream(stream)))
    return g


def _bwd_logit_strides(lam_logits, B, n, G):
    """Strides of the logits as the V2 backward takes them: [B, n, Hq/2], [B, Hq/2] or [Hq/2]."""
    f32 = torch.float32
    if lam_logits.dim() == 3:
        _need(lam_logits, "lam_logits", f32, (B, n, G))
        return n * G, G
    if lam_logits.dim() == 2:
        _need(lam_logits, "lam_logits", f32, (B, G))
        return G, 0
    _need(lam_logits, "lam_logits", f32, (G,))
    return 0, 0


def diffattn_v2_forward_train(q, k, v, lam_logits, causal: bool = True, softmax_scale: float = 0.0, out=None,
                              saved=None, stream=None):
    """diffattn_v2_forward (bf16, d = 128) that also saves each row's lse and O_1, O_2 for
    diffattn_v2_backward_saved; lam_logits [B, n, Hq/2], [B, Hq/2] or [Hq/2].  Returns (out, saved)."""
    B, n, Hq, d = q.shape
    Hkv = k.shape[2]
    _need(q, "q", torch.bfloat16, (B, n, Hq, d))
    _need(k, "k", torch.bfloat16, (B, n, Hkv, d))
    _need(v, "v", torch.bfloat16, (B, n, Hkv, d))
    G = Hq // 2
    sb, st = _bwd_logit_strides(lam_logits, B, n, G)
    if out is None:
        out = torch.empty((B, n, G, d), device=q.device, dtype=torch.bfloat16)
    _need(out, "out", torch.bfloat16, (B, n, G, d))
    need = v2_forward_saved_bytes(B, Hq, n, d)
    saved = _saved_buf(saved, need, q.device)
    _check(lib().diffattn_v2_forward_train(B, Hq, Hkv, n, d, _ptr(q), _ptr(k), _ptr(v), _ptr(lam_logits), sb, st,
                                           float(softmax_scale), 1 if causal else 0, _ptr(out), _ptr(saved),
                                           saved.numel(), _stream(stream)))
    return out, saved


def diffattn_v2_backward_saved(q, k, v, lam_logits, dy, saved, causal: bool = True, softmax_scale: float = 0.0,
                               workspace=None, stream=None) -> dict:
    """diffattn_v2_backward (bf16, d = 128) from the `saved` of diffattn_v2_forward_train on the same inputs."""
    B, n, Hq, d = q.shape
    Hkv = k.shape[2]
    for name, t, shp in (("q", q, (B, n, Hq, d)), ("k", k, (B, n, Hkv, d)), ("v", v, (B, n, Hkv, d)),
                         ("dy", dy, (B, n, Hq // 2, d))):
        _need(t, name, torch.bfloat16, shp)
    G = Hq // 2
    sb, st = _bwd_logit_strides(lam_logits, B, n, G)
    need = v2_backward_workspace_bytes(B, Hq, n, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    wp, wn = _ws_args(workspace, need)
    f32 = torch.float32
    g = {"dq": torch.empty(q.shape, device=q.device, dtype=f32), "dk": torch.empty(k.shape, device=q.device, dtype=f32),
         "dv": torch.empty(v.shape, device=q.device, dtype=f32), "dlogits": torch.empty_like(lam_logits)}
    _check(lib().diffattn_v2_backward_saved(B, Hq, Hkv, n, d, _ptr(q), _ptr(k), _ptr(v), _ptr(lam_logits), sb, st,
                                            float(softmax_scale), 1 if causal else 0, _ptr(dy), _ptr(saved),
                                            saved.numel(), _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]),
                                            _ptr(g["dlogits"]), wp, wn, _stream(stream)))
    return g


def lambda_reparam_backward(lq1, lk1, lq2, lk2, dlam, stream=None):
    """Gradients of lambda_reparam's lambda with respect to lq1, lk1, lq2, lk2, given dlam [1] (device)."""
    for name, t in (("lq1", lq1), ("lk1", lk1), ("lq2", lq2), ("lk2", lk2)):
        _need(t, name, torch.float32, (lq1.numel(),))
    _need(dlam, "dlam", torch.float32, (1,))
    outs = [torch.empty_like(t) for t in (lq1, lk1, lq2, lk2)]
    _check(lib().lambda_reparam_backward(_ptr(lq1), _ptr(lk1), _ptr(lq2), _ptr(lk2), lq1.numel(), _ptr(dlam),
                                         *(_ptr(o) for o in outs), _stream(stream)))
    return tuple(outs)


def _logit_strides(lam_logits, B, n, G):
    if lam_logits.shape == (G,):
        return 0, 0
    if lam_logits.shape == (n, G):
        return 0, G
    if lam_logits.shape == (B, n, G):
        return n * G, G
    raise ValueError(f"lam_logits must be [Hq/2], [n, Hq/2] or [B, n, Hq/2]; got {tuple(lam_logits.shape)}")


def diffattn_v2_forward_fp8qk(q, k, scales, v, lam_logits, causal: bool = True, softmax_scale: float = 0.0,
                              out=None, stream=None) -> torch.Tensor:
    """DIFF V2 forward with e4m3 queries and keys (QK^T on the FP8 tensor-core path).

    q: [B, n, Hq, 128], k: [B, n, Hkv, 128] e4m3 codes (torch.float8_e4m3fn or their bytes as uint8)
    of Q / q_scale and K / k_scale; scales = (q_scale, k_scale); v bf16 [B, n, Hkv, 128]; lam_logits
    as for diffattn_v2_forward.  The result is diffattn_v2_forward's for Q = q_scale e4m3(q),
    K = k_scale e4m3(k).  Returns out [B, n, Hq/2, 128] bf16.
    """
    B, n, Hq, d = q.shape
    Hkv = k.shape[2]
    _need_fp8(q, "q", (B, n, Hq, d))
    _need_fp8(k, "k", (B, n, Hkv, d))
    _need(v, "v", torch.bfloat16, (B, n, Hkv, d))
    G = Hq // 2
    _need(lam_logits, "lam_logits", torch.float32)
    sb, st = _logit_strides(lam_logits, B, n, G)
    if out is None:
        out = torch.empty((B, n, G, d), device=v.device, dtype=torch.bfloat16)
    _need(out, "out", torch.bfloat16, (B, n, G, d))
    qs, ks = (float(x) for x in scales)
    _check(lib().diffattn_v2_forward_fp8qk(B, Hq, Hkv, n, d, _ptr(q), _ptr(k), qs, ks, _ptr(v), _ptr(lam_logits),
                                           sb, st, float(softmax_scale), 1 if causal else 0, _ptr(out),
                                           _stream(stream)))
    return out


def diffattn_v2_forward(q, k, v, lam_logits, causal: bool = True, softmax_scale: float = 0.0, out=None,
                        stream=None) -> torch.Tensor:
    """DIFF V2 forward: out_g = attn[2g] - sigmoid(logit) attn[2g+1]; BSHD tensors.

    q: [B, n, Hq, d]; k, v: [B, n, Hkv, d]; lam_logits: fp32 [Hq/2] (one per
    pair), [n, Hq/2] or [B, n, Hq/2].  Returns out [B, n, Hq/2, d].
    """
    B, n, Hq, d = q.shape
    Hkv = k.shape[2]
    dt = q.dtype
    _need(q, "q", dt)
    _need(k, "k", dt, (B, n, Hkv, d))
    _need(v, "v", dt, (B, n, Hkv, d))
    G = Hq // 2
    _need(lam_logits, "lam_logits", torch.float32)
    sb, st = _logit_strides(lam_logits, B, n, G)
    if out is None:
        out = torch.empty((B, n, G, d), device=q.device, dtype=dt)
    _need(out, "out", dt, (B, n, G, d))
    _check(lib().diffattn_v2_forward(_dt(q), B, Hq, Hkv, n, d, _ptr(q), _ptr(k), _ptr(v), _ptr(lam_logits),
                                     sb, st, float(softmax_scale), 1 if causal else 0, _ptr(out),
                                     _stream(stream)))
    return out


def projection(a, w, out=None, stream=None) -> torch.Tensor:
    """out = a w^T on the tensor cores: a [M, K], w [N, K] (bf16; K, N multiples of 8) -> [M, N] bf16."""
    M, K = a.shape
    N = w.shape[0]
    _need(a, "a", torch.bfloat16, (M, K))
    _need(w, "w", torch.bfloat16, (N, K))
    if out is None:
        out = torch.empty((M, N), device=a.device, dtype=torch.bfloat16)
    _need(out, "out", torch.bfloat16, (M, N))
    _check(lib().diffattn_projection(M, N, K, _ptr(a), _ptr(w), _ptr(out), _stream(stream)))
    return out


def layer_workspace_bytes(B: int, n: int, H: int, d: int) -> int:
    return int(lib().diffattn_layer_workspace(B, n, H, d))


def layer_forward(x, w_qkv, w_o, lq1, lk1, lq2, lk2, lambda_init_value: float, H: int, gamma=None,
                  eps: float = 1e-5, causal: bool = True, out=None, workspace=None, stream=None) -> torch.Tensor:
    """DIFF V1 attention layer: X [W^Q | W^K | W^V], the operator with the per-head norm, W^O.

    x: [B, n, D] bf16; w_qkv: [3 H 2d, D] bf16 (rows: W^Q's columns, then W^K's, then W^V's; head i's
    2d columns of W^Q hold Q_1 then Q_2); w_o: [D, H 2d] bf16; lq1..lk2: fp32 [d]; gamma: fp32 [2d] or
    None.  workspace: a device tensor of layer_workspace_bytes(B, n, H, d) bytes (allocated here if
    None).  Returns out [B, n, D] bf16.
    """
    B, n, D = x.shape
    d = w_qkv.shape[0] // (6 * H)
    _need(x, "x", torch.bfloat16, (B, n, D))
    _need(w_qkv, "w_qkv", torch.bfloat16, (6 * H * d, D))
    _need(w_o, "w_o", torch.bfloat16, (D, 2 * H * d))
    for name, t in (("lq1", lq1), ("lk1", lk1), ("lq2", lq2), ("lk2", lk2)):
        _need(t, name, torch.float32, (d,))
    if gamma is not None:
        _need(gamma, "gamma", torch.float32, (2 * d,))
    if out is None:
        out = torch.empty((B, n, D), device=x.device, dtype=torch.bfloat16)
    _need(out, "out", torch.bfloat16, (B, n, D))
    need = layer_workspace_bytes(B, n, H, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    wp, wn = _ws_args(workspace, need)
    _check(lib().diffattn_layer_forward(B, n, D, H, d, _ptr(x), _ptr(w_qkv), _ptr(w_o), _ptr(lq1), _ptr(lk1),
                                        _ptr(lq2), _ptr(lk2), float(lambda_init_value), _ptr(gamma), float(eps),
                                        1 if causal else 0, _ptr(out), wp, wn, _stream(stream)))
    return out


def v2_layer_workspace_bytes(B: int, n: int, Hq: int, Hkv: int, d: int) -> int:
    return int(lib().diffattn_v2_layer_workspace(B, n, Hq, Hkv, d))


def v2_layer_forward(x, w_qkvl, w_o, Hq: int, Hkv: int, causal: bool = True, out=None, workspace=None,
                     stream=None) -> torch.Tensor:
    """DIFF V2 attention layer: X [W^Q | W^K | W^V | W^lambda], the V2 operator, W^O.

    x: [B, n, D] bf16; w_qkvl: [(Hq + 2 Hkv) d + Hq/2, D] bf16 (rows: W^Q's columns, W^K's, W^V's,
    then the Hq/2 pair-logit columns of W^lambda); w_o: [D, Hq/2 d] bf16.  Returns out [B, n, D].
    """
    B, n, D = x.shape
    G = Hq // 2
    d = (w_qkvl.shape[0] - G) // (Hq + 2 * Hkv)
    _need(x, "x", torch.bfloat16, (B, n, D))
    _need(w_qkvl, "w_qkvl", torch.bfloat16, ((Hq + 2 * Hkv) * d + G, D))
    _need(w_o, "w_o", torch.bfloat16, (D, G * d))
    if out is None:
        out = torch.empty((B, n, D), device=x.device, dtype=torch.bfloat16)
    _need(out, "out", torch.bfloat16, (B, n, D))
    need = v2_layer_workspace_bytes(B, n, Hq, Hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    wp, wn = _ws_args(workspace, need)
    _check(lib().diffattn_v2_layer_forward(B, n, D, Hq, Hkv, d, _ptr(x), _ptr(w_qkvl), _ptr(w_o),
                                           1 if causal else 0, _ptr(out), wp, wn, _stream(stream)))
    return out


def bounds_checked() -> bool:
    """True when the loaded library is the bounds-check build."""
    return bool(lib().diffattn_bounds_checked())


def debug_bounds_selftest(stream=None) -> None:
    """Bounds-check build: one checked store out of its limit (skipped and recorded)."""
    _check(lib().diffattn_debug_bounds_selftest(_stream(stream)))


def debug_item_plan(grid: int, units: int, nqt: int, qt0: int, n: int, causal: bool, kv_unit_bytes: int):
    """The host's item plan of a persistent d = 128 forward: (first [grid + 1], items [units nqt]) as
    numpy uint16 arrays, or None when the launch is too large for a plan."""
    import numpy as np
    first = np.zeros(max(grid, 0) + 1, dtype=np.uint16)
    items = np.zeros(max(units * nqt, 1), dtype=np.uint16)
    cnt = lib().diffattn_debug_item_plan(grid, units, nqt, qt0, n, 1 if causal else 0, kv_unit_bytes,
                                         first.ctypes.data_as(ctypes.c_void_p), items.ctypes.data_as(ctypes.c_void_p))
    return None if cnt == 0 else (first, items)


def device_status(stream=None) -> int:
    """Synchronise the stream, read and clear the device status word (raises on error)."""
    st = lib().diffattn_device_status(_stream(stream))
    _check(st)
    return st


def debug_wait_timeout(budget_ns: int, stream=None) -> None:
    """Launch the bounded-wait self-test kernel (its wait must run out)."""
    _check(lib().diffattn_debug_wait_timeout(int(budget_ns), _stream(stream)))


def launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(lib().diffattn_launch_count())
