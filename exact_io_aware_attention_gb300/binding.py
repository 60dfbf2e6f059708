"""Thin Python binding of libfa.so (include/fa.h).

Argument marshalling only: tensors are checked, their device pointers, strides
and the current CUDA stream are handed to the C ABI, and the status code is
turned into an exception. Every step of the computation runs in the library's CUDA
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

FA_BF16, FA_F32, FA_F16 = 0, 1, 2
_DTYPES = {torch.bfloat16: FA_BF16, torch.float32: FA_F32, torch.float16: FA_F16}


class FaTensor(ctypes.Structure):
    """struct fa_tensor: one [B, H, rows, d] operand with element strides."""
    _fields_ = [("data", ctypes.c_void_p), ("stride_b", ctypes.c_int64),
                ("stride_h", ctypes.c_int64), ("stride_n", ctypes.c_int64),
                ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32)]


# Every symbol include/fa.h declares, with its ctypes signature.
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_tp = ctypes.POINTER(FaTensor)
SIGNATURES = {
    "fa_abi_version": ([], _i),
    "fa_status_string": ([_i], ctypes.c_char_p),
    "fa_last_error": ([], ctypes.c_char_p),
    "fa_forward": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _vp], _i),
    "fa_forward_f32": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _vp], _i),
    "fa_forward_ex": ([_tp, _tp, _tp, _tp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp, _vp], _i),
    "fa_forward_split_ex": ([_tp, _tp, _tp, _tp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp, _i, _vp,
                             _sz, _vp], _i),
    "fa_forward_split_workspace_bytes": ([_i, _i, _i, _i, _i], _sz),
    "fa_forward_num_splits": ([_i, _i, _i, _i, _i, _i], _i),
    "fa_backward_workspace_bytes": ([_i, _i, _i, _i], _sz),
    "fa_backward_min_workspace_bytes": ([_i, _i, _i, _i], _sz),
    "fa_backward_one_pass_workspace_bytes": ([_i, _i, _i, _i], _sz),
    "fa_backward": ([_vp] * 9 + [_i, _i, _i, _i, _i, _f, _vp, _vp, _sz, _vp], _i),
    "fa_backward_ex": ([_tp] * 5 + [_vp] + [_tp] * 3 +
                       [_i, _i, _i, _i, _i, _i, _f, _vp, _vp, _sz, _vp], _i),
    "fa_backward_noalloc": ([_vp] * 9 + [_i, _i, _i, _i, _i, _f, _vp, _vp], _i),
    "fa_backward_noalloc_max_bytes": ([], _sz),
    "fa_device_status": ([_vp, ctypes.POINTER(ctypes.c_uint)], _i),
    "fa_debug_configure": ([ctypes.c_uint, ctypes.c_ulonglong], _i),
    "fa_num_kernels": ([], _i),
    "fa_kernel_name": ([_i], ctypes.c_char_p),
    "fa_profile_enable": ([_i], _i),
    "fa_profile_collect": ([ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int), _i], _i),
    "fa_measure_exp2_rate": ([ctypes.POINTER(ctypes.c_double)], _i),
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


def _lib_fast():
    return _lib if _lib is not None else load_library()


def _check(status: int, what: str):
    if status != FA_OK:
        detail = load_library().fa_last_error().decode()
        raise FAError(status, what, detail)


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(device=None):
    """The current CUDA stream of `device` (default: the current device) as a
    raw handle."""
    if _raw_stream is not None:
        idx = device.index if device is not None and device.index is not None else \
            torch.cuda.current_device()
        return ctypes.c_void_p(_raw_stream(idx))
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _desc(t, name):
    """fa_tensor of a [B, H, rows, d] CUDA tensor whose d elements are contiguous."""
    dt = _DTYPES.get(t.dtype)
    st = t.stride()
    if not t.is_cuda or len(st) != 4 or dt is None or (st[3] != 1 and t.shape[3] > 1):
        raise ValueError(f"{name} must be a 4-D CUDA tensor [B, H, rows, d] of a supported "
                         f"dtype with contiguous rows (got {tuple(t.shape)}, {t.dtype}, {st})")
    return FaTensor(t.data_ptr(), st[0], st[1], st[2], dt, 0)


def _shapes(q, kv, qlike=()):
    """(B, H, Nq, Nk, d) of q [B,H,Nq,d] and k, v [B,H,Nk,d]."""
    qs = q.shape
    if len(qs) != 4:
        raise ValueError("q must be [B, H, Nq, d]")
    B, H, Nq, d = qs
    ks = kv[0].shape
    Nk = ks[2] if len(ks) == 4 else -1
    for t in kv:
        ts = t.shape
        if len(ts) != 4 or ts[0] != B or ts[1] != H or ts[2] != Nk or ts[3] != d:
            raise ValueError("k and v must be [B, H, Nk, d] with q's B, H and d")
    for t in qlike:
        if t.shape != qs:
            raise ValueError("o and do must have q's shape")
    return B, H, Nq, Nk, d


def _mask(block_mask, nq, nk):
    if block_mask is None:
        return None
    tq, tk = -(-nq // 128), -(-nk // 128)
    if (not block_mask.is_cuda or block_mask.dtype != torch.uint8 or
            tuple(block_mask.shape) != (tq, tk) or not block_mask.is_contiguous()):
        raise ValueError(f"block_mask must be a contiguous uint8 CUDA tensor [{tq}, {tk}]")
    return block_mask


def default_num_splits(B, H, Nq, Nk, d, causal, device=None) -> int:
    """The library's choice of key splits for the forward pass of this shape
    (1: no split) on ``device`` (default: the current CUDA device)."""
    dev = torch.device(device) if device is not None else None
    if dev is None or dev.index is None or dev.index == torch.cuda.current_device():
        return int(load_library().fa_forward_num_splits(B, H, Nq, Nk, d, int(bool(causal))))
    with torch.cuda.device(dev):
        return int(load_library().fa_forward_num_splits(B, H, Nq, Nk, d, int(bool(causal))))


_sm_counts = {}


def _fills_gpu(B, H, Nq, d, device) -> bool:
    """Whether the plain forward's grid (one CTA per pair of 128-row query
    tiles and head; one per tile for d = 256) already gives every SM a CTA,
    so no split can help."""
    idx = device.index if device.index is not None else torch.cuda.current_device()
    sms = _sm_counts.get(idx)
    if sms is None:
        sms = _sm_counts[idx] = torch.cuda.get_device_properties(idx).multi_processor_count
    tiles = -(-Nq // 128)
    return (tiles if d == 256 else (tiles + 1) // 2) * B * H >= sms


def forward(q, k, v, causal: bool = False, scale: float | None = None, block_mask=None,
            out=None, lse=None, o_dtype=None, num_splits: int | None = None):
    """O, LSE = attention(q, k, v).

    q is [B, H, Nq, d], k and v [B, H, Nk, d], all bf16 or all fp16, with any
    strides over the first three dimensions (e.g. permuted views of
    [B, N, H, d] tensors); d is 64, 96, 128 or 256. O has q's shape and, unless
    ``out`` is given, q's layout and dtype (or ``o_dtype=torch.float32``);
    LSE is fp32 contiguous [B, H, Nq]. With ``causal``, query i sees key j
    iff j <= i + Nk - Nq.

    ``num_splits``: how many CTAs share the keys of one query tile (their
    partial results are merged by a second kernel). None lets the library
    choose: 1 unless the query tiles alone would leave SMs idle, as when
    decoding against a long cache.
    """
    B, H, Nq, Nk, d = _shapes(q, (k, v))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    mask = _mask(block_mask, Nq, Nk)
    if out is None:
        out = torch.empty_like(q, dtype=q.dtype if o_dtype is None else o_dtype)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or lse.shape != (B, H, Nq) or \
            lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("out must be [B, H, Nq, d] and lse contiguous fp32 [B, H, Nq]")
    dq_, dk_, dv_, do_ = _desc(q, "q"), _desc(k, "k"), _desc(v, "v"), _desc(out, "out")
    lib = _lib_fast()
    if num_splits is None:
        num_splits = 1 if _fills_gpu(B, H, Nq, d, q.device) else \
            default_num_splits(B, H, Nq, Nk, d, causal, q.device)
    if num_splits == 1:
        _check(lib.fa_forward_ex(
            ctypes.byref(dq_), ctypes.byref(dk_), ctypes.byref(dv_), ctypes.byref(do_),
            _ptr(lse), B, H, Nq, Nk, d, int(bool(causal)), scale, _ptr(mask),
            _stream(q.device)), "fa_forward_ex")
        return out, lse
    nbytes = int(lib.fa_forward_split_workspace_bytes(B, H, Nq, d, int(num_splits)))
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    _check(lib.fa_forward_split_ex(
        ctypes.byref(dq_), ctypes.byref(dk_), ctypes.byref(dv_), ctypes.byref(do_), _ptr(lse),
        B, H, Nq, Nk, d, int(bool(causal)), scale, _ptr(mask), int(num_splits), _ptr(ws),
        nbytes, _stream(q.device)), "fa_forward_split_ex")
    return out, lse


def backward_workspace_bytes(B, H, N, d, algo: str = "auto") -> int:
    """Workspace bytes of the backward pass for N query rows per (batch, head),
    which select its form: the faster form for the head dimension ("auto"),
    the one-pass kernel ("fused", d <= 128), or the row statistics only, the
    two-kernel form ("split")."""
    lib = _lib_fast()
    if algo == "split":
        return int(lib.fa_backward_min_workspace_bytes(B, H, N, d))
    if algo == "fused":
        n = int(lib.fa_backward_one_pass_workspace_bytes(B, H, N, d))
        if n == 0 and B * H * N > 0:
            raise ValueError(f"the one-pass backward supports d <= 128, not {d}")
        return n
    if algo != "auto":
        raise ValueError(f"algo must be 'auto', 'fused' or 'split', not {algo!r}")
    return int(lib.fa_backward_workspace_bytes(B, H, N, d))


def backward(q, k, v, o, do, lse, causal: bool = False, scale: float | None = None,
             block_mask=None, workspace=None, dq=None, dk=None, dv=None, algo: str = "auto"):
    """dQ, dK, dV of attention for upstream gradient ``do``.

    Shapes and layouts as in ``forward``: q, o, do, dq are [B, H, Nq, d], k, v,
    dk, dv [B, H, Nk, d], all bf16 or all fp16, with any strides over the
    first three dimensions; each gradient takes its input's layout unless
    given. ``algo`` sizes the workspace when none is given, which selects the
    form: "auto" (the faster form for the head dimension: one-pass for
    d <= 96), "fused" (the one-pass backward, d <= 128; dQ accumulated with
    atomic adds) or "split" (the two-kernel form, bitwise reproducible). A
    given ``workspace`` decides by its size, as fa_backward_ex does.
    """
    B, H, Nq, Nk, d = _shapes(q, (k, v), (o, do))
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    mask = _mask(block_mask, Nq, Nk)
    nbytes = backward_workspace_bytes(B, H, Nq, d, algo)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if dq.shape != q.shape or dk.shape != k.shape or dv.shape != v.shape:
        raise ValueError("dq, dk, dv must have the shapes of q, k, v")
    if lse.shape != (B, H, Nq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [B, H, Nq]")
    r = [ctypes.byref(_desc(t, n)) for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"),
                                                (do, "do"), (dq, "dq"), (dk, "dk"), (dv, "dv"))]
    _check(_lib_fast().fa_backward_ex(
        r[0], r[1], r[2], r[3], r[4], _ptr(lse), r[5], r[6], r[7], B, H, Nq, Nk, d,
        int(bool(causal)), scale, _ptr(mask), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(q.device)), "fa_backward_ex")
    return dq, dk, dv


def device_status(stream=None) -> int:
    """Synchronise and read/clear the device status word (0 = no wait gave up)."""
    code = ctypes.c_uint(0)
    st = _stream() if stream is None else ctypes.c_void_p(stream)
    rc = load_library().fa_device_status(st, ctypes.byref(code))
    if rc not in (FA_OK, 5):
        raise FAError(rc, "fa_device_status")
    return int(code.value)


def measure_exp2_rate() -> float:
    """ex2.approx operations per second of the whole current device, at the
    clocks of the moment (a measurement, run once; synchronises)."""
    r = ctypes.c_double(0.0)
    _check(_lib_fast().fa_measure_exp2_rate(ctypes.byref(r)), "fa_measure_exp2_rate")
    return float(r.value)


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
        if do.stride(3) != 1:
            do = do.contiguous()
        dq, dk, dv = backward(q, k, v, o, do, lse, causal=ctx.causal, scale=ctx.scale,
                              block_mask=ctx.block_mask)
        return dq, dk, dv, None, None, None


def attention(q, k, v, causal: bool = False, scale: float | None = None, block_mask=None):
    """Differentiable exact attention (autograd wrapper around forward/backward)."""
    return _Attention.apply(q, k, v, causal, scale, block_mask)
