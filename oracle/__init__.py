"""fp64 CPU oracle for exact scaled dot-product attention.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the CPU-baseline
leg of ``bench.py`` use it. The product path never imports this package, and
this package never imports the product package; the two share only the seeded
input generators, which hold none of the method's arithmetic.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, pthreads); this
module compiles it with gcc and marshals numpy arrays to it. Every function
takes and returns float64 arrays: queries, outputs and their gradients laid out
``[B, H, Nq, d]``, keys and values ``[B, H, Nk, d]``, statistics ``[B, H, Nq]``.

What is computed, and which passage of the pages each part follows, is stated
at the top of ``attn_oracle.c``; ``merge`` / ``merge_lse`` (numpy, below) are
the pages' rule for combining the softmax results of disjoint key blocks. Parity status: every entry point is pinned by
``tests/test_oracle_*.py`` (worked examples printed on the pages, closed forms,
invariants, brute force and finite differences).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into oracle/_build/liboracle.so (gcc, -O2, IEEE)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
             "-fno-fast-math", "-ffp-contract=off", "-Wall", "-Wextra",
             "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int)
            up = ctypes.POINTER(ctypes.c_ubyte)
            i = ctypes.c_int
            lib.oracle_forward.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, i,
                                           ctypes.c_double, up, i, ip, i, i]
            lib.oracle_forward.restype = i
            lib.oracle_forward_tiled.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, i,
                                                 ctypes.c_double, up, i, i, i, i]
            lib.oracle_forward_tiled.restype = i
            lib.oracle_backward.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i,
                                            i, ctypes.c_double, up, i, ip, i, ip, i, i]
            lib.oracle_backward.restype = i
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _f64(x, name):
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    if a.ndim != 4:
        raise ValueError(f"{name} must be [B, H, N, d], got shape {a.shape}")
    return a


def _ptr(a, ctype=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _mask(block_mask, Nq, Nk, mask_tile):
    if block_mask is None:
        return None
    m = np.ascontiguousarray(np.asarray(block_mask, dtype=np.uint8))
    Tq, Tk = (Nq + mask_tile - 1) // mask_tile, (Nk + mask_tile - 1) // mask_tile
    if m.shape != (Tq, Tk):
        raise ValueError(f"block_mask must be [{Tq}, {Tk}] for Nq={Nq}, Nk={Nk}, "
                         f"tile={mask_tile}")
    return m


def _shapes(q, kv, extra=()):
    """(B, H, Nq, Nk, d) of queries q [B,H,Nq,d] and keys/values [B,H,Nk,d]."""
    B, H, Nq, d = q.shape
    Nk = kv[0].shape[2]
    if any(t.shape != (B, H, Nk, d) for t in kv):
        raise ValueError("k and v must be [B, H, Nk, d] with q's B, H and d")
    if any(t.shape != q.shape for t in extra):
        raise ValueError("do must have q's shape")
    return B, H, Nq, Nk, d


def _idx(rows, N):
    if rows is None:
        return None
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    if r.ndim != 1 or (r.size and (r.min() < 0 or r.max() >= N)):
        raise ValueError("row indices out of range")
    return r


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what} failed with code {rc}")


def forward(q, k, v, causal=False, scale=None, block_mask=None, mask_tile=128, rows=None,
            threads=None):
    """Exact attention from the definition: returns (O, LSE) in float64.

    q is ``[B, H, Nq, d]``, k and v ``[B, H, Nk, d]``. ``rows`` (optional)
    restricts the computation to those query rows; the outputs are then
    ``[B, H, len(rows), d]`` and ``[B, H, len(rows)]``.
    """
    q, k, v = _f64(q, "q"), _f64(k, "k"), _f64(v, "v")
    B, H, Nq, Nk, d = _shapes(q, (k, v))
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    m = _mask(block_mask, Nq, Nk, mask_tile)
    r = _idx(rows, Nq)
    nr = Nq if r is None else r.size
    o = np.empty((B, H, nr, d), np.float64)
    lse = np.empty((B, H, nr), np.float64)
    if B * H * nr == 0:
        return o, lse
    rc = _load().oracle_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk,
                                d, int(bool(causal)), scale, _ptr(m, ctypes.c_ubyte), mask_tile,
                                _ptr(r, ctypes.c_int), nr, threads or default_threads())
    _check(rc, "oracle_forward")
    return o, lse


def forward_tiled(q, k, v, causal=False, scale=None, block_mask=None, mask_tile=128, bq=64,
                  bk=64, threads=None):
    """The online-softmax recurrence over bq x bk blocks: returns (O, LSE)."""
    q, k, v = _f64(q, "q"), _f64(k, "k"), _f64(v, "v")
    B, H, Nq, Nk, d = _shapes(q, (k, v))
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    m = _mask(block_mask, Nq, Nk, mask_tile)
    o = np.empty((B, H, Nq, d), np.float64)
    lse = np.empty((B, H, Nq), np.float64)
    if B * H * Nq == 0:
        return o, lse
    rc = _load().oracle_forward_tiled(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq,
                                      Nk, d, int(bool(causal)), scale, _ptr(m, ctypes.c_ubyte),
                                      mask_tile, int(bq), int(bk), threads or default_threads())
    _check(rc, "oracle_forward_tiled")
    return o, lse


def backward(q, k, v, do, causal=False, scale=None, block_mask=None, mask_tile=128,
             qrows=None, kcols=None, want_dq=True, want_dkv=True, threads=None):
    """Analytic gradients of exact attention for upstream gradient ``do``.

    q and do are ``[B, H, Nq, d]``, k and v ``[B, H, Nk, d]``. Returns a dict
    with ``dq`` ([B,H,nq,d]), ``dk``/``dv`` ([B,H,nk,d]), and ``lse``/``D``
    ([B,H,Nq], the row statistics the oracle computed itself).
    ``qrows``/``kcols`` restrict dq / dk,dv to those rows.
    """
    q, k, v, do = _f64(q, "q"), _f64(k, "k"), _f64(v, "v"), _f64(do, "do")
    B, H, Nq, Nk, d = _shapes(q, (k, v), (do,))
    scale = 1.0 / np.sqrt(d) if scale is None else float(scale)
    m = _mask(block_mask, Nq, Nk, mask_tile)
    # a non-NULL index array with count 0 tells the C side to skip that part
    qr = _idx(qrows, Nq) if want_dq else np.zeros(1, np.int32)
    kc = _idx(kcols, Nk) if want_dkv else np.zeros(1, np.int32)
    nq = Nq if qr is None else (qr.size if want_dq else 0)
    nk = Nk if kc is None else (kc.size if want_dkv else 0)
    dq = np.empty((B, H, nq, d), np.float64)
    dk = np.empty((B, H, nk, d), np.float64)
    dv = np.empty((B, H, nk, d), np.float64)
    lse = np.empty((B, H, Nq), np.float64)
    D = np.empty((B, H, Nq), np.float64)
    if B * H * Nq > 0:
        rc = _load().oracle_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), _ptr(dk),
                                     _ptr(dv), _ptr(lse), _ptr(D), B, H, Nq, Nk, d,
                                     int(bool(causal)), scale, _ptr(m, ctypes.c_ubyte),
                                     mask_tile, _ptr(qr, ctypes.c_int), nq,
                                     _ptr(kc, ctypes.c_int), nk, threads or default_threads())
        _check(rc, "oracle_backward")
    return {"dq": dq, "dk": dk, "dv": dv, "lse": lse, "D": D}


def merge(o_parts, m_parts, l_parts):
    """Merge of per-block softmax results over disjoint key blocks, folding the
    two-block rule of "Paper Notes: FlashAttention", section "Tiling:
    Block-by-Block Softmax", left to right:

        m = max(m1, m2),  l = e^(m1 - m) l1 + e^(m2 - m) l2,

    with each block's output rescaled by the same factor as its sum:
    O = (e^(m1 - m) l1 O1 + e^(m2 - m) l2 O2) / l. O_s is block s's normalised
    output [..., d], m_s and l_s its row max and row sum [...]; a block in which
    a row sees no key has m_s = -inf, l_s = 0 and contributes nothing.
    Returns (O, m, l), float64; a row with no key anywhere gets O = 0,
    m = -inf, l = 0.
    """
    o = np.asarray(o_parts[0], np.float64)
    m = np.asarray(m_parts[0], np.float64)
    l = np.asarray(l_parts[0], np.float64)
    acc = o * l[..., None]  # unnormalised output of the blocks merged so far
    for o2, m2, l2 in zip(o_parts[1:], m_parts[1:], l_parts[1:]):
        o2 = np.asarray(o2, np.float64)
        m2 = np.asarray(m2, np.float64)
        l2 = np.asarray(l2, np.float64)
        m_new = np.maximum(m, m2)
        with np.errstate(invalid="ignore"):
            a1 = np.where(np.isneginf(m), 0.0, np.exp(m - m_new))
            a2 = np.where(np.isneginf(m2), 0.0, np.exp(m2 - m_new))
        l = a1 * l + a2 * l2
        acc = a1[..., None] * acc + (a2 * l2)[..., None] * o2
        m = m_new
    with np.errstate(invalid="ignore", divide="ignore"):
        out = np.where((l > 0)[..., None], acc / np.where(l > 0, l, 1.0)[..., None], 0.0)
    return out, m, l


def merge_lse(o_parts, lse_parts):
    """``merge`` for blocks summarised by LSE_s = m_s + ln l_s (the form the
    library stores): each block enters as (O_s, m = LSE_s, l = 1), or
    (0, -inf, 0) when LSE_s = -inf. Returns (O, LSE)."""
    lse_parts = [np.asarray(x, np.float64) for x in lse_parts]
    ls = [np.where(np.isneginf(x), 0.0, 1.0) for x in lse_parts]
    o, m, l = merge(o_parts, lse_parts, ls)
    with np.errstate(divide="ignore"):
        lse = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return o, lse
