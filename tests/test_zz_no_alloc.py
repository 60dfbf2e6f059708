"""fa_backward_noalloc: the backward pass for callers that cannot allocate
device memory where they run it (a plug-in inside an application that owns
all device memory, a runtime that forbids allocating after start-up). Such a
caller cannot hand fa_backward a workspace, so this entry point uses a fixed
scratch area built into the library.

The GPU test calls it through the C ABI, twice in a row on different shapes
(the second call reuses the area the first one left behind). The kernels see
the same inputs as fa_backward with a caller-allocated workspace, so dK and dV
must equal that call's bit for bit, and so must dQ where the two-kernel form
runs (head dimension 256); the one-pass form (the default for 64 to 128) sums
dQ with fp32 atomics, so there dQ must agree to one bf16 ulp. The first call is also held to the fp64
oracle. The device's free memory is read before and after
each call: a call that allocated would change it. This file is collected last
so that a run stopping at its first failure has already run every other
test."""
import ctypes

import numpy as np
import pytest
import torch

from exact_io_aware_attention_gb300 import binding
from exact_io_aware_attention_gb300 import build as fa_build
from exact_io_aware_attention_gb300 import inputs as gen
import oracle
from parity import assert_same_up_to_atomics, check_grad, f64


@pytest.fixture(scope="module")
def lib():
    fa_build.build()
    return binding.load_library()


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    """Validation happens before any CUDA call, so this runs without a GPU."""
    fake = ctypes.c_void_p(0x10000)
    B, H, N, d = 512, 64, 8192, 128  # 2^28 query rows: 2 GiB of row statistics
    assert lib.fa_backward_workspace_bytes(B, H, N, d) > lib.fa_backward_noalloc_max_bytes()
    rc = lib.fa_backward_noalloc(*([fake] * 9), B, H, N, d, 1, 0.088, None, None)
    assert rc == 2  # FA_ERR_UNSUPPORTED
    msg = lib.fa_last_error().decode()
    assert "needs" in msg and str(lib.fa_backward_noalloc_max_bytes()) in msg
    assert lib.fa_backward_noalloc(*([None] * 9), B, H, N, d, 1, 0.088, None, None) == 1


@pytest.mark.gpu
def test_noalloc_backward_matches_workspace_backward(lib):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cases = [((1, 4, 1024, 128), True, None), ((2, 2, 768, 64), False, 0.2),
             ((1, 2, 700, 256), True, None)]
    for n, (shape, causal, scale) in enumerate(cases):
        B, H, N, d = shape
        assert lib.fa_backward_workspace_bytes(B, H, N, d) <= lib.fa_backward_noalloc_max_bytes()
        scale = 1.0 / np.sqrt(d) if scale is None else scale
        inp = gen.make_inputs(B, H, N, d, case=900 + n)
        q, k, v, do = (inp[t].cuda() for t in ("q", "k", "v", "do"))
        o, lse = binding.forward(q, k, v, causal=causal, scale=scale)
        ref = binding.backward(q, k, v, o, do, lse, causal=causal, scale=scale)
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        rc = lib.fa_backward_noalloc(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq),
                                     _p(dk), _p(dv), B, H, N, d, int(causal), scale, None, stream)
        assert rc == 0, lib.fa_last_error().decode()
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info()[0]
        assert binding.device_status() == 0
        assert free_after == free_before, \
            f"call {n + 1}: free device memory went from {free_before} to {free_after} bytes"
        for name, got, want in (("dk", dk, ref[1]), ("dv", dv, ref[2])):
            assert torch.equal(got, want), f"call {n + 1}: {name} differs from fa_backward"
        if d > 128:  # the two-kernel form (the only form there): bit for bit
            assert torch.equal(dq, ref[0]), f"call {n + 1}: dq differs from fa_backward"
        else:  # the one-pass backward sums dQ with fp32 atomics: one bf16 ulp
            assert_same_up_to_atomics(dq, ref[0], f"call {n + 1}: dq against fa_backward")
        if n == 0:
            sl = lambda t: f64(t[:1, :1])
            g = oracle.backward(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(inp["do"]),
                                causal=causal, scale=scale)
            for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
                check_grad(f64(got[0, 0]), g[name][0, 0], name, "fa_backward_noalloc")
