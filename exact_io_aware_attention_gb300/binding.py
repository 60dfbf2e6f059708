"""Thin Python binding of libfa.so (include/fa.h).

Argument marshalling only: tensors are checked, their device pointers and the
current CUDA stream are handed to the C ABI, and the status code is turned
into an exception. Every step of the computation runs in the library's CUDA
kernels; PyTorch only provides device memory and streams. There is no CPU or
fallback path: if libfa.so is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfa.so")

FA_OK = 0
STATUS_NAMES = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED",
                3: "FA_ERR_MISALIGNED", 4: "FA_ERR_CUDA", 5: "FA_ERR_TIMEOUT"}

# Every symbol include/fa.h declares, with its ctypes signature.
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "fa_abi_version": ([], _i),
    "fa_status_string": ([_i], ctypes.c_char_p),
    "fa_last_error": ([], ctypes.c_char_p),
    "fa_forward": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _vp], _i),
    "fa_forward_f32": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _vp], _i),
    "fa_backward_workspace_bytes": ([_i, _i, _i, _i], _sz),
    "fa_backward": ([_vp] * 9 + [_i, _i, _i, _i, _i, _f, _vp, _vp, _sz, _vp], _i),
    "fa_backward_noalloc": ([_vp] * 9 + [_i, _i, _i, _i, _i, _f, _vp, _vp], _i),
    "fa_backward_noalloc_max_bytes": ([], _sz),
    "fa_device_status": ([_vp, ctypes.POINTER(ctypes.c_uint)], _i),
    "fa_debug_configure": ([ctypes.c_uint, ctypes.c_ulonglong], _i),
    "fa_num_kernels": ([], _i),
    "fa_kernel_name": ([_i], ctypes.c_char_p),
    "fa_profile_enable": ([_i], _i),
    "fa_profile_collect": ([ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int), _i], _i),
}

_lock = threading.Lock()
_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        msg = f"{what}: {STATUS_NAMES.get(status, status)}"
        super().__init__(msg + (f" ({detail})" if detail else ""))


def load_library(path: str | None = None):
    """Load libfa.so (built by ``exact_io_aware_attention_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(
                    f"{p} is missing: build the CUDA library first "
                    "(python -m exact_io_aware_attention_gb300.build)")
            lib = ctypes.CDLL(p)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            if path is not None:
                return lib
            _lib = lib
    return _lib


def _check(status: int, what: str):
    if status != FA_OK:
        detail = load_library().fa_last_error().decode() if status == 4 else ""
        raise FAError(status, what, detail)


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _check_qkv(*ts):
    q = ts[0]
    if q.dim() != 4:
        raise ValueError("tensors must be [B, H, N, d]")
    for t in ts:
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("tensors must be contiguous bf16 CUDA tensors")
        if t.shape != q.shape:
            raise ValueError("tensors must share one shape")
    return q.shape


def _mask(block_mask, n):
    if block_mask is None:
        return None
    t = -(-n // 128)
    if (not block_mask.is_cuda or block_mask.dtype != torch.uint8 or
            tuple(block_mask.shape) != (t, t) or not block_mask.is_contiguous()):
        raise ValueError(f"block_mask must be a contiguous uint8 CUDA tensor [{t}, {t}]")
    return block_mask


def forward(q, k, v, causal: bool = False, scale: float | None = None, block_mask=None,
            out=None, lse=None, o_dtype=torch.bfloat16):
    """O, LSE = attention(q, k, v): O [B,H,N,d] (bf16, or fp32 with
    ``o_dtype=torch.float32``), LSE fp32 [B,H,N]."""
    B, H, N, d = _check_qkv(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    mask = _mask(block_mask, N)
    if out is None:
        out = torch.empty((B, H, N, d), dtype=o_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fn = load_library().fa_forward_f32 if out.dtype == torch.float32 else load_library().fa_forward
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d, int(bool(causal)),
              scale, _ptr(mask), _stream()), "fa_forward")
    return out, lse


def backward_workspace_bytes(B, H, N, d) -> int:
    return int(load_library().fa_backward_workspace_bytes(B, H, N, d))


def backward(q, k, v, o, do, lse, causal: bool = False, scale: float | None = None,
             block_mask=None, workspace=None, dq=None, dk=None, dv=None):
    """dQ, dK, dV of attention for upstream gradient ``do`` (all bf16 [B,H,N,d])."""
    B, H, N, d = _check_qkv(q, k, v, o, do)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    mask = _mask(block_mask, N)
    nbytes = backward_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(load_library().fa_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
        B, H, N, d, int(bool(causal)), scale, _ptr(mask), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream()), "fa_backward")
    return dq, dk, dv


def device_status(stream=None) -> int:
    """Synchronise and read/clear the device status word (0 = no wait gave up)."""
    code = ctypes.c_uint(0)
    st = _stream() if stream is None else ctypes.c_void_p(stream)
    rc = load_library().fa_device_status(st, ctypes.byref(code))
    if rc not in (FA_OK, 5):
        raise FAError(rc, "fa_device_status")
    return int(code.value)


def profile_enable(enable: bool = True):
    """Bracket every kernel launch with CUDA events on its stream (no sync)."""
    _check(load_library().fa_profile_enable(int(bool(enable))), "fa_profile_enable")


def profile_collect() -> dict:
    """{kernel name: (total ms, launches)} since the last collect; synchronises
    on the recorded events."""
    lib = load_library()
    n = lib.fa_num_kernels()
    ms = (ctypes.c_float * n)()
    cnt = (ctypes.c_int * n)()
    _check(lib.fa_profile_collect(ms, cnt, n), "fa_profile_collect")
    return {lib.fa_kernel_name(k).decode(): (float(ms[k]), int(cnt[k])) for k in range(n)}


class _Attention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, causal, scale, block_mask):
        o, lse = forward(q, k, v, causal=causal, scale=scale, block_mask=block_mask)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal, ctx.scale, ctx.block_mask = causal, scale, block_mask
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = backward(q, k, v, o, do.contiguous(), lse, causal=ctx.causal,
                              scale=ctx.scale, block_mask=ctx.block_mask)
        return dq, dk, dv, None, None, None


def attention(q, k, v, causal: bool = False, scale: float | None = None, block_mask=None):
    """Differentiable exact attention (autograd wrapper around forward/backward)."""
    return _Attention.apply(q, k, v, causal, scale, block_mask)
