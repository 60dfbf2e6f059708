"""Extra device memory of the long-context workload: B=1, H=16, N=65536,
d=128, causal.

The method stores only O and the per-row softmax statistics and recomputes
the score tiles in the backward pass, so its extra memory is O(N) instead of
the O(N^2) of the score matrix ("Paper Notes: FlashAttention", "Experiments &
Results"; aicassindra page "FlashAttention", "O(N) memory: the footprint that
unlocks long context"). Here the caller allocates every buffer up front: the
inputs Q, K, V, dO, the outputs O, dQ, dK, dV, the fp32 LSE and the backward
workspace. The test runs one forward and one backward through the C ABI and
checks that

  - the library allocates nothing: the device's free memory
    (cudaMemGetInfo) and the caching allocator's peak are unchanged across
    the two calls;
  - the extra memory beyond the inputs and outputs is exactly the LSE plus
    fa_backward_workspace_bytes, which is linear in N (it is printed beside
    the bytes a 16-bit score matrix would need).

The default (one-pass) backward's workspace holds an fp32 dQ accumulator,
4d bytes per query row; a second backward with fa_backward_min_workspace_bytes
(the two-kernel form, 8 bytes per row) shows the smallest footprint, again
without any allocation.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_attention_gb300 import binding
from exact_io_aware_attention_gb300 import inputs as gen
from parity import check_lse, f64

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def test_long_context_extra_memory_is_lse_plus_workspace():
    lib = binding.load_library()
    w = gen.WORKLOADS["long_context_n65536"]
    B, H, N, d = w.B, w.H, w.N, w.d
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    # the same kernels on a small shape first, so that loading their code
    # (lazy module loading) happens outside the measured calls
    small = gen.make_inputs(1, 2, 256, d, case=950)
    qs, ks, vs, dos = (small[t].cuda() for t in ("q", "k", "v", "do"))
    os_, lses = binding.forward(qs, ks, vs, causal=True, scale=w.scale)
    binding.backward(qs, ks, vs, os_, dos, lses, causal=True, scale=w.scale)

    inp = gen.make_workload_inputs(w)
    q, k, v, do = (inp[t].cuda() for t in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    ws_bytes = lib.fa_backward_workspace_bytes(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    io_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, do, o, dq, dk, dv))
    extra_bytes = lse.numel() * 4 + ws_bytes

    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    allocated0 = torch.cuda.memory_allocated()
    free0 = torch.cuda.mem_get_info()[0]
    rc = lib.fa_forward(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, N, d, 1, w.scale, None,
                        stream)
    assert rc == 0, lib.fa_last_error().decode()
    rc = lib.fa_backward(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk), _p(dv),
                         B, H, N, d, 1, w.scale, None, _p(ws), ws_bytes, stream)
    assert rc == 0, lib.fa_last_error().decode()
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    peak = torch.cuda.max_memory_allocated()
    assert binding.device_status() == 0

    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    assert peak == allocated0, f"the caching allocator grew by {peak - allocated0} bytes"
    # the two-kernel form with the smallest workspace (a prefix of the same buffer)
    min_bytes = lib.fa_backward_min_workspace_bytes(B, H, N, d)
    dq2 = torch.empty_like(q)
    torch.cuda.synchronize()
    free2 = torch.cuda.mem_get_info()[0]
    rc = lib.fa_backward(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq2), _p(dk), _p(dv),
                         B, H, N, d, 1, w.scale, None, _p(ws), min_bytes, stream)
    assert rc == 0, lib.fa_last_error().decode()
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free2
    assert binding.device_status() == 0
    rel = float((dq2.float() - dq.float()).norm() / dq.float().norm())
    assert rel < 1e-3, f"the two backward forms disagree on dQ: rel-L2 {rel:.2e}"
    # O(N) extra memory: 4 bytes of LSE plus the workspace's bytes per query
    # row, against 2 N bytes per row for a 16-bit score matrix
    rows = B * H * N
    assert extra_bytes <= rows * 4 + ws_bytes
    s_bytes = rows * N * 2
    per_row = extra_bytes / rows
    assert per_row <= 4 + 8 + 4 * d + 1, f"{per_row:.1f} extra bytes per query row"
    print(f"\nlong-context extra memory: inputs+outputs {io_bytes / 1e9:.3f} GB; "
          f"LSE {lse.numel() * 4 / 1e6:.1f} MB + workspace {ws_bytes / 1e6:.1f} MB = "
          f"{extra_bytes / 1e6:.1f} MB ({per_row:.1f} B per query row); with the smallest "
          f"workspace (two-kernel form) {(lse.numel() * 4 + min_bytes) / 1e6:.1f} MB "
          f"({(lse.numel() * 4 + min_bytes) / rows:.1f} B per row); "
          f"a 16-bit score matrix would be {s_bytes / 1e9:.1f} GB; "
          f"cudaMemGetInfo free before/after {free0}/{free1}")

    # the results of the measured calls are the method's: LSE on sampled rows
    # against the oracle, finite gradients
    assert torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all()
    rows_s = np.array([0, 1, 127, 128, 4097, N - 1], dtype=np.int32)
    sl = lambda t: f64(t[0:1, 3:4])
    _, lse_ref = oracle.forward(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), causal=True,
                                scale=w.scale, rows=rows_s)
    check_lse(f64(lse[0:1, 3:4])[..., rows_s], lse_ref, "long-context LSE")
