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
    assert lib.fa_abi_version() == 2
    for code, name in binding.STATUS_NAMES.items():
        assert lib.fa_status_string(code).decode() == name
    assert lib.fa_status_string(99).decode() == "FA_ERR_UNKNOWN"


def test_workspace_bytes(lib):
    """Row statistics D and LSE*log2(e) (fp32, padded to whole 128-row query
    tiles per (batch, head)); the one-pass backward adds an fp32 dQ accumulator
    of d floats per padded row. The default size is the faster form's: the
    one-pass form for d <= 128, the two-kernel form (statistics only) at 256."""
    up = lambda x: (x + 255) // 256 * 256
    B, H, N = 4, 16, 4096
    rows = B * H * N
    stats = 2 * up(4 * rows)
    for d in (64, 96, 128):
        assert lib.fa_backward_workspace_bytes(B, H, N, d) == stats + up(4 * rows * d)
        assert lib.fa_backward_one_pass_workspace_bytes(B, H, N, d) == stats + up(4 * rows * d)
    assert lib.fa_backward_workspace_bytes(B, H, N, 256) == stats
    assert lib.fa_backward_one_pass_workspace_bytes(B, H, N, 256) == 0
    for d in (64, 96, 128, 256):
        assert lib.fa_backward_min_workspace_bytes(B, H, N, d) == stats
    padded = 3 * 5 * 256
    assert lib.fa_backward_workspace_bytes(3, 5, 129, 64) == 2 * up(4 * padded) + up(4 * padded * 64)
    assert lib.fa_backward_min_workspace_bytes(3, 5, 129, 64) == 2 * up(4 * padded)
    assert lib.fa_backward_workspace_bytes(1, 1, 1, 256) == 2 * up(4 * 128)
    for f in (lib.fa_backward_workspace_bytes, lib.fa_backward_min_workspace_bytes,
              lib.fa_backward_one_pass_workspace_bytes):
        assert f(-1, 1, 128, 64) == 0
        assert f(1, 1, 0, 64) == 0


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
    (dict(d=80), UNSUPPORTED), (dict(d=512), UNSUPPORTED), (dict(N=65537), UNSUPPORTED),
    (dict(N=128 * 513), UNSUPPORTED),
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


# -- strided descriptors and separate query / key lengths ---------------------

def desc(ptr=A, sb=None, sh=None, sn=64, dtype=binding.FA_BF16, reserved=0, H=2, N=300, d=64):
    sh = N * d if sh is None else sh
    sb = H * N * d if sb is None else sb
    return binding.FaTensor(ptr.value if ptr is not None else None, sb, sh, sn, dtype, reserved)


def fwd_ex(lib, q=None, k=None, v=None, o=None, lse=B_, B=1, H=2, Nq=300, Nk=300, d=64,
           causal=1):
    q = q or desc(N=Nq, H=H, d=d, sn=d)
    k = k or desc(N=Nk, H=H, d=d, sn=d)
    v = v or desc(N=Nk, H=H, d=d, sn=d)
    o = o or desc(ptr=B_, N=Nq, H=H, d=d, sn=d)
    return lib.fa_forward_ex(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.byref(o),
                             lse, B, H, Nq, Nk, d, causal, 0.125, None, None)


# statuses that mean "the arguments passed every host check": the call then
# fails at the device check (fake pointers: no GPU here, or not device memory)
PASSED_HOST_CHECKS = (INVALID, 4)


@pytest.mark.parametrize("case,status", [
    (dict(q=desc(sn=60)), MISALIGNED),                   # row stride 120 bytes
    (dict(k=desc(sh=300 * 64 + 4)), MISALIGNED),          # head stride not 16-byte aligned
    (dict(v=desc(sn=-64)), UNSUPPORTED),                  # negative stride
    (dict(q=desc(sn=0)), UNSUPPORTED),                    # zero stride of a long dimension
    (dict(q=desc(sn=1 << 40)), UNSUPPORTED),              # beyond the tensor-map range
    (dict(q=desc(dtype=3)), UNSUPPORTED),                 # an element type the kernels lack
    (dict(q=desc(dtype=binding.FA_F16)), UNSUPPORTED),    # f16 Q with bf16 K and V
    (dict(q=desc(dtype=binding.FA_F32)), UNSUPPORTED),    # fp32 inputs
    (dict(o=desc(ptr=B_, dtype=7)), UNSUPPORTED),
    (dict(q=desc(reserved=1)), INVALID),
    (dict(q=desc(ptr=None)), INVALID),
    (dict(q=desc(ptr=M)), MISALIGNED),
    (dict(Nk=0), UNSUPPORTED),
    (dict(Nq=-1), INVALID),
    (dict(Nk=65537), UNSUPPORTED),
])
def test_forward_ex_rejects_bad_descriptors(lib, case, status):
    assert fwd_ex(lib, **case) == status


@pytest.mark.parametrize("case", [
    dict(),                                                        # contiguous, N = 300
    dict(Nq=1, Nk=4097),                                           # one query, ragged keys
    dict(Nq=1000, Nk=129),
    dict(q=desc(sn=2 * 64, sh=64, sb=300 * 2 * 64)),               # [B, N, H, d] layout
    dict(o=desc(ptr=B_, dtype=binding.FA_F32, sn=64, sh=300 * 64)),  # fp32 O
    dict(B=1, q=desc(sb=3)),                                       # stride of a length-1 dim
    dict(d=96),                                                    # head dimension 96
    dict(q=desc(dtype=binding.FA_F16), k=desc(dtype=binding.FA_F16),  # fp16 throughout
         v=desc(dtype=binding.FA_F16), o=desc(ptr=B_, dtype=binding.FA_F16)),
    dict(q=desc(dtype=binding.FA_F16), k=desc(dtype=binding.FA_F16),  # fp16 in, fp32 O
         v=desc(dtype=binding.FA_F16), o=desc(ptr=B_, dtype=binding.FA_F32)),
])
def test_forward_ex_accepts_general_shapes(lib, case):
    assert fwd_ex(lib, **case) in PASSED_HOST_CHECKS


def test_forward_ex_empty_queries_is_noop(lib):
    assert fwd_ex(lib, Nq=0) == OK
    assert lib.fa_forward_ex(None, None, None, None, None, 1, 1, 0, 128, 64, 0, 0.1, None,
                             None) == OK


def test_backward_ex_checks_every_operand(lib):
    ws_bytes = lib.fa_backward_workspace_bytes(1, 2, 300, 64)
    good = [desc() for _ in range(8)]
    for k in range(8):
        ds = list(good)
        ds[k] = desc(sn=12)
        r = [ctypes.byref(x) for x in ds]
        st = lib.fa_backward_ex(r[0], r[1], r[2], r[3], r[4], B_, r[5], r[6], r[7], 1, 2, 300,
                                300, 64, 1, 0.125, None, B_, ws_bytes, None)
        assert st == MISALIGNED, k
    r = [ctypes.byref(x) for x in good]
    # below the row statistics' size (the two-kernel form's minimum)
    min_bytes = lib.fa_backward_min_workspace_bytes(1, 2, 300, 64)
    assert lib.fa_backward_ex(r[0], r[1], r[2], r[3], r[4], B_, r[5], r[6], r[7], 1, 2, 300, 300,
                              64, 1, 0.125, None, B_, min_bytes - 256, None) == INVALID
    o32 = desc(dtype=binding.FA_F32)
    assert lib.fa_backward_ex(r[0], r[1], r[2], ctypes.byref(o32), r[4], B_, r[5], r[6], r[7], 1,
                              2, 300, 300, 64, 1, 0.125, None, B_, ws_bytes, None) == UNSUPPORTED


# -- the forward with the keys split over several CTAs ------------------------

def test_split_workspace_bytes(lib):
    up = lambda x: (x + 255) // 256 * 256
    assert lib.fa_forward_split_workspace_bytes(2, 8, 1, 128, 9) == \
        up(9 * 2 * 8 * 1 * 128 * 4) + up(9 * 2 * 8 * 1 * 4)
    assert lib.fa_forward_split_workspace_bytes(2, 8, 1, 128, 1) == 0
    assert lib.fa_forward_split_workspace_bytes(2, 8, 1, 128, 0) == 0
    assert lib.fa_forward_split_workspace_bytes(-1, 8, 1, 128, 4) == 0


def test_num_splits_without_a_device_is_one(lib):
    # no GPU here: the library cannot read the SM count and declines to split
    assert lib.fa_forward_num_splits(1, 16, 1, 65536, 128, 1) == 1
    assert lib.fa_forward_num_splits(1, 16, 0, 65536, 128, 1) == 1


def split_fwd(lib, ns, ws=B_, ws_bytes=None, Nq=1, Nk=4096, d=128):
    q = desc(N=Nq, d=d, sn=d)
    k = desc(N=Nk, d=d, sn=d)
    o = desc(ptr=B_, N=Nq, d=d, sn=d)
    if ws_bytes is None:
        ws_bytes = lib.fa_forward_split_workspace_bytes(1, 2, Nq, d, max(ns, 1))
    return lib.fa_forward_split_ex(ctypes.byref(q), ctypes.byref(k), ctypes.byref(k),
                                   ctypes.byref(o), B_, 1, 2, Nq, Nk, d, 1, 0.1, None, ns, ws,
                                   ws_bytes, None)


def test_split_forward_rejects_bad_arguments(lib):
    assert split_fwd(lib, 0) == INVALID
    assert split_fwd(lib, -3) == INVALID
    assert split_fwd(lib, 129) == UNSUPPORTED
    assert split_fwd(lib, 4, ws=None) == INVALID
    assert split_fwd(lib, 4, ws_bytes=1024) == INVALID
    assert split_fwd(lib, 4, ws=ctypes.c_void_p(0x20010)) == MISALIGNED
    assert split_fwd(lib, 4) in PASSED_HOST_CHECKS
    assert split_fwd(lib, 1, ws=None, ws_bytes=0) in PASSED_HOST_CHECKS  # no split: no workspace


def test_head_dim_256_passes_host_checks(lib):
    assert fwd_ex(lib, d=256) in PASSED_HOST_CHECKS
    assert bwd(lib, d=256) in PASSED_HOST_CHECKS
    assert lib.fa_backward_noalloc(A, A, A, A, A, A, B_, B_, B_, 1, 1, 256, 256, 0, 0.1, None,
                                   None) in PASSED_HOST_CHECKS
    assert bwd(lib, d=192) == UNSUPPORTED
