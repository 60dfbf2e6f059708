"""The C ABI without a GPU: the library loads, exports every function
include/fa.h declares, and rejects bad arguments on the host with the
documented status codes before any CUDA call is made."""
import ctypes
import os
import re

import pytest

from exact_io_aware_attention_gb300 import binding
from exact_io_aware_attention_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")

OK, INVALID, UNSUPPORTED, MISALIGNED = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return binding.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 7
    for n in names:
        assert hasattr(lib, n), f"{n} declared in fa.h but not exported"
        assert n in binding.SIGNATURES, f"{n} has no binding signature"


def test_status_strings(lib):
    assert lib.fa_abi_version() == 1
    for code, name in binding.STATUS_NAMES.items():
        assert lib.fa_status_string(code).decode() == name
    assert lib.fa_status_string(99).decode() == "FA_ERR_UNKNOWN"


def test_workspace_bytes(lib):
    B, H, N, d = 4, 16, 4096, 128
    rows = B * H * N
    up = lambda x: (x + 255) // 256 * 256
    assert lib.fa_backward_workspace_bytes(B, H, N, d) == 2 * up(4 * rows)
    assert lib.fa_backward_workspace_bytes(-1, 1, 128, 64) == 0
    assert lib.fa_backward_workspace_bytes(1, 1, 0, 64) == 0


A = ctypes.c_void_p(0x10000)     # fake 16-byte aligned addresses: never dereferenced,
B_ = ctypes.c_void_p(0x20000)    # every call below fails validation first
M = ctypes.c_void_p(0x30008)     # 8-byte aligned only


def fwd(lib, q=A, k=A, v=A, o=B_, lse=B_, B=1, H=1, N=256, d=64, causal=0, scale=0.125):
    return lib.fa_forward(q, k, v, o, lse, B, H, N, d, causal, scale, None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), INVALID), (dict(o=None), INVALID), (dict(lse=None), INVALID),
    (dict(B=-1), INVALID), (dict(N=-128), INVALID), (dict(d=0), INVALID),
    (dict(scale=0.0), INVALID), (dict(scale=-1.0), INVALID), (dict(scale=float("inf")), INVALID),
    (dict(scale=float("nan")), INVALID),
    (dict(d=96), UNSUPPORTED), (dict(d=256), UNSUPPORTED), (dict(N=100), UNSUPPORTED),
    (dict(N=129), UNSUPPORTED), (dict(N=128 * 513), UNSUPPORTED),
    (dict(B=65536, H=256, N=256), UNSUPPORTED),
    (dict(q=M), MISALIGNED), (dict(v=M), MISALIGNED), (dict(lse=M), MISALIGNED),
])
def test_forward_rejects_bad_arguments(lib, kw, status):
    assert fwd(lib, **kw) == status


def test_forward_empty_is_noop_without_touching_memory(lib):
    assert fwd(lib, q=None, k=None, v=None, o=None, lse=None, N=0) == OK
    assert fwd(lib, B=0) == OK
    assert lib.fa_forward_f32(None, None, None, None, None, 3, 0, 128, 64, 1, 0.1, None,
                              None) == OK


def bwd(lib, ws=B_, ws_bytes=None, dq=B_, d=64, N=256, B=1, H=1):
    if ws_bytes is None:
        ws_bytes = lib.fa_backward_workspace_bytes(B, H, N, d)
    return lib.fa_backward(A, A, A, A, A, A, dq, B_, B_, B, H, N, d, 0, 0.125, None, ws,
                           ws_bytes, None)


def test_backward_rejects_bad_arguments(lib):
    assert bwd(lib, ws=None) == INVALID
    assert bwd(lib, ws_bytes=1024) == INVALID
    assert bwd(lib, dq=None) == INVALID
    assert bwd(lib, dq=M) == MISALIGNED
    assert bwd(lib, ws=ctypes.c_void_p(0x20010)) == MISALIGNED  # 16-B but not 256-B aligned
    assert bwd(lib, d=80) == UNSUPPORTED
    assert bwd(lib, N=0) == OK


def test_binding_refuses_to_run_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        binding.load_library(str(tmp_path / "libfa.so"))
