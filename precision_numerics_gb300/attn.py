"""Python binding of libattn.so (ctypes): argument marshalling only.

Every function here checks tensor metadata, allocates outputs with PyTorch
when the caller does not pass them, and calls the C entry point of the same
name; all arithmetic runs in the library's CUDA kernels.  There is no CPU
fallback: if the library is missing or a call fails, an exception is raised.

Tensors are [B, H, N, d], contiguous, on the current CUDA device, either all
torch.bfloat16 (tensor-core path) or all torch.float32 (reference mode).
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from . import build as _build

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT = range(5)
ATTN_DTYPE_BF16, ATTN_DTYPE_FP32 = 0, 1

EXPORTED = ("attn_version", "attn_status_string", "attn_last_error", "attn_fwd",
            "attn_bwd_workspace_bytes", "attn_bwd", "attn_bwd_preprocess", "attn_bwd_main",
            "attn_bwd_dq_convert", "attn_check_status", "attn_selftest_wait_timeout",
            "attn_bwd_noalloc", "attn_fwd_stable", "attn_quantize_int8", "attn_fwd_int8",
            "attn_quantize_int8_as_bf16", "attn_fwd_int8_as_bf16")


class AttnError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str):
        self.status = status
        super().__init__(f"{fn} failed: {_status_string(status)}"
                         + (f" -- {detail}" if detail else ""))


_LIB = None
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t

_SIGNATURES = {
    "attn_version": (_i, []),
    "attn_status_string": (ctypes.c_char_p, [_i]),
    "attn_last_error": (ctypes.c_char_p, []),
    "attn_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _i, _vp]),
    "attn_bwd_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "attn_bwd": (_i, [_vp] * 9 + [_i, _i, _i, _i, _f, _i, _i, _vp, _sz, _vp]),
    "attn_bwd_preprocess": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _sz, _vp]),
    "attn_bwd_main": (_i, [_vp] * 6 + [_i, _i, _i, _i, _f, _i, _i, _vp, _sz, _vp]),
    "attn_bwd_dq_convert": (_i, [_vp, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp]),
    "attn_check_status": (_i, [_vp]),
    "attn_selftest_wait_timeout": (_i, [ctypes.c_ulonglong, _vp]),
    "attn_bwd_noalloc": (_i, [_vp] * 9 + [_i, _i, _i, _i, _f, _i, _vp]),
    "attn_fwd_stable": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _f, _i, _vp]),
    "attn_quantize_int8": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "attn_fwd_int8": (_i, [_vp] * 7 + [_i, _i, _i, _i, _f, _i, _vp]),
    "attn_quantize_int8_as_bf16": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "attn_fwd_int8_as_bf16": (_i, [_vp] * 7 + [_i, _i, _i, _i, _f, _i, _vp]),
}


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libattn.so (built by precision_numerics_gb300.build.build())."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    path = path or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first "
                           "(python -m precision_numerics_gb300.build)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path == _build.LIB:
        _LIB = lib
    return lib


def _status_string(status: int) -> str:
    try:
        return load_library().attn_status_string(status).decode()
    except Exception:  # noqa: BLE001 - only used to format an error
        return f"status {status}"


def _call(name: str, *args) -> int:
    lib = load_library()
    status = getattr(lib, name)(*args)
    if status != ATTN_OK:
        raise AttnError(name, status, lib.attn_last_error().decode())
    return status


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return ATTN_DTYPE_BF16
    if t.dtype == torch.float32:
        return ATTN_DTYPE_FP32
    raise TypeError(f"attention tensors must be bfloat16 or float32, got {t.dtype}")


def _check_bhnd(name: str, t: torch.Tensor, shape=None, dtype=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != 4:
        raise ValueError(f"{name} must be [B, H, N, d], got shape {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")


def _check_lse(lse, B, H, N):
    if tuple(lse.shape) != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor")


def _default_scale(d: int, scale):
    return 1.0 / math.sqrt(d) if scale is None else float(scale)


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


def attn_version() -> int:
    return int(load_library().attn_version())


def attn_fwd(q, k, v, scale=None, causal=False, o=None, lse=None, stream=None):
    """O, LSE = attention forward.  Returns (o, lse)."""
    _check_bhnd("q", q)
    B, H, N, d = q.shape
    for name, t in (("k", k), ("v", v)):
        _check_bhnd(name, t, q.shape, q.dtype)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_bhnd("o", o, q.shape, q.dtype)
    _check_lse(lse, B, H, N)
    _call("attn_fwd", q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
          B, H, N, d, _default_scale(d, scale), int(bool(causal)), _dtype_code(q), _stream(stream))
    return o, lse


def attn_fwd_stable(q, k, v, scale=None, causal=False, beta=2.0, o=None, lse=None, stream=None):
    """Forward with the stabilised normaliser (beta * repeated row max).  Returns (o, lse)."""
    _check_bhnd("q", q, dtype=torch.bfloat16)
    B, H, N, d = q.shape
    for name, t in (("k", k), ("v", v)):
        _check_bhnd(name, t, q.shape, q.dtype)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_bhnd("o", o, q.shape, q.dtype)
    _check_lse(lse, B, H, N)
    _call("attn_fwd_stable", q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
          lse.data_ptr(), B, H, N, d, _default_scale(d, scale), int(bool(causal)), float(beta),
          ATTN_DTYPE_BF16, _stream(stream))
    return o, lse


def attn_quantize_int8(x, codes=None, scales=None, stream=None):
    """Per-token symmetric INT8 codes and FP32 scales of a BF16 [B,H,N,d] tensor."""
    _check_bhnd("x", x, dtype=torch.bfloat16)
    B, H, N, d = x.shape
    if codes is None:
        codes = torch.empty(x.shape, dtype=torch.int8, device=x.device)
    if scales is None:
        scales = torch.empty((B, H, N), dtype=torch.float32, device=x.device)
    _check_bhnd("codes", codes, x.shape, torch.int8)
    _check_lse(scales, B, H, N)
    _call("attn_quantize_int8", x.data_ptr(), codes.data_ptr(), scales.data_ptr(), B, H, N, d,
          _stream(stream))
    return codes, scales


def attn_fwd_int8(q8, q_scale, k8, k_scale, v, scale=None, causal=False, o=None, lse=None,
                  stream=None):
    """Forward on per-token INT8 Q and K (attn_quantize_int8) and BF16 V.  Returns (o, lse)."""
    _check_bhnd("v", v, dtype=torch.bfloat16)
    B, H, N, d = v.shape
    for name, t in (("q8", q8), ("k8", k8)):
        _check_bhnd(name, t, v.shape, torch.int8)
    _check_lse(q_scale, B, H, N)
    _check_lse(k_scale, B, H, N)
    if o is None:
        o = torch.empty_like(v)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=v.device)
    _check_bhnd("o", o, v.shape, v.dtype)
    _check_lse(lse, B, H, N)
    _call("attn_fwd_int8", q8.data_ptr(), q_scale.data_ptr(), k8.data_ptr(), k_scale.data_ptr(),
          v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d, _default_scale(d, scale),
          int(bool(causal)), _stream(stream))
    return o, lse


def int8_scale_rows(N: int) -> int:
    """Rows per head of the padded scale layout of the *_as_bf16 INT8 calls (N rounded up to 128)."""
    return (N + 127) // 128 * 128


def _check_padded_scales(name, t, B, H, N):
    if (tuple(t.shape) != (B, H, int8_scale_rows(N)) or t.dtype != torch.float32
            or not t.is_contiguous() or not t.is_cuda):
        raise ValueError(f"{name} must be a contiguous float32 CUDA tensor [B, H, {int8_scale_rows(N)}]")


def attn_quantize_int8_as_bf16(x, codes=None, scales=None, stream=None):
    """attn_quantize_int8 with the codes held in BF16 and the scales padded to [B, H, N_pad]."""
    _check_bhnd("x", x, dtype=torch.bfloat16)
    B, H, N, d = x.shape
    if codes is None:
        codes = torch.empty_like(x)
    if scales is None:
        scales = torch.empty((B, H, int8_scale_rows(N)), dtype=torch.float32, device=x.device)
    _check_bhnd("codes", codes, x.shape, torch.bfloat16)
    _check_padded_scales("scales", scales, B, H, N)
    _call("attn_quantize_int8_as_bf16", x.data_ptr(), codes.data_ptr(), scales.data_ptr(), B, H, N,
          d, _stream(stream))
    return codes, scales


def attn_fwd_int8_as_bf16(q_codes, q_scale, k_codes, k_scale, v, scale=None, causal=False, o=None,
                          lse=None, stream=None):
    """attn_fwd_int8 on BF16-held codes (attn_quantize_int8_as_bf16), on the tcgen05 path."""
    _check_bhnd("v", v, dtype=torch.bfloat16)
    B, H, N, d = v.shape
    for name, t in (("q_codes", q_codes), ("k_codes", k_codes)):
        _check_bhnd(name, t, v.shape, torch.bfloat16)
    _check_padded_scales("q_scale", q_scale, B, H, N)
    _check_padded_scales("k_scale", k_scale, B, H, N)
    if o is None:
        o = torch.empty_like(v)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=v.device)
    _check_bhnd("o", o, v.shape, v.dtype)
    _check_lse(lse, B, H, N)
    _call("attn_fwd_int8_as_bf16", q_codes.data_ptr(), q_scale.data_ptr(), k_codes.data_ptr(),
          k_scale.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
          _default_scale(d, scale), int(bool(causal)), _stream(stream))
    return o, lse


def attn_bwd_workspace_bytes(B: int, H: int, N: int, d: int, dtype=torch.bfloat16) -> int:
    code = ATTN_DTYPE_BF16 if dtype == torch.bfloat16 else ATTN_DTYPE_FP32
    return int(load_library().attn_bwd_workspace_bytes(B, H, N, d, code))


def _workspace(q, workspace):
    B, H, N, d = q.shape
    need = attn_bwd_workspace_bytes(B, H, N, d, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if _nbytes(workspace) < need:
        raise ValueError(f"workspace too small: {_nbytes(workspace)} bytes, {need} needed")
    return workspace


def attn_bwd(q, k, v, o, lse, do, scale=None, causal=False, dq=None, dk=None, dv=None,
             workspace=None, stream=None):
    """dQ, dK, dV of L = sum(dO o O) from the saved LSE.  Returns (dq, dk, dv)."""
    _check_bhnd("q", q)
    B, H, N, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o), ("do", do)):
        _check_bhnd(name, t, q.shape, q.dtype)
    _check_lse(lse, B, H, N)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_bhnd(name, t, q.shape, q.dtype)
    ws = _workspace(q, workspace)
    _call("attn_bwd", q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
          do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
          _default_scale(d, scale), int(bool(causal)), _dtype_code(q), ws.data_ptr(), _nbytes(ws),
          _stream(stream))
    return dq, dk, dv


def attn_bwd_preprocess(o, lse, do, workspace, stream=None):
    """Phase 1 of the BF16 backward (delta, LSE*log2(e), zeroed dQ accumulator)."""
    B, H, N, d = o.shape
    _call("attn_bwd_preprocess", o.data_ptr(), lse.data_ptr(), do.data_ptr(), B, H, N, d,
          _dtype_code(o), workspace.data_ptr(), _nbytes(workspace), _stream(stream))


def attn_bwd_main(q, k, v, do, dk, dv, workspace, scale=None, causal=False, stream=None):
    """Phase 2 of the BF16 backward (dK, dV and the dQ accumulation)."""
    B, H, N, d = q.shape
    _call("attn_bwd_main", q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(),
          dk.data_ptr(), dv.data_ptr(), B, H, N, d, _default_scale(d, scale), int(bool(causal)),
          _dtype_code(q), workspace.data_ptr(), _nbytes(workspace), _stream(stream))


def attn_bwd_dq_convert(dq, workspace, scale=None, stream=None):
    """Phase 3 of the BF16 backward (dQ = bf16(scale * accumulator))."""
    B, H, N, d = dq.shape
    _call("attn_bwd_dq_convert", dq.data_ptr(), B, H, N, d, _default_scale(d, scale),
          _dtype_code(dq), workspace.data_ptr(), _nbytes(workspace), _stream(stream))


def attn_check_status(stream=None) -> None:
    """Synchronize and raise AttnError if a kernel gave up on a bounded wait."""
    _call("attn_check_status", _stream(stream))


def attn_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    """Enqueue the bounded-wait self-test kernel (see include/attn.h)."""
    _call("attn_selftest_wait_timeout", int(limit_ns), _stream(stream))


def attn_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, scale=None, causal=False, stream=None):
    """attn_bwd for callers that must not allocate device memory: BF16 only,
    outputs passed in, scratch taken from the library's fixed 32 MiB array
    (see include/attn.h for the size limit and the sharing rules)."""
    _check_bhnd("q", q, dtype=torch.bfloat16)
    B, H, N, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o), ("do", do), ("dq", dq), ("dk", dk), ("dv", dv)):
        _check_bhnd(name, t, q.shape, q.dtype)
    _check_lse(lse, B, H, N)
    _call("attn_bwd_noalloc", q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
          lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
          _default_scale(d, scale), int(bool(causal)), _stream(stream))
    return dq, dk, dv
