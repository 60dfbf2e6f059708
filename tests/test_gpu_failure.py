"""Failure detection on the GPU without a fault. With FA_DEBUG_SKIP_LOADS the
TMA producers issue no copy, so the kernels' barrier waits are never satisfied.
Each wait gives up after a short limit; the kernel records kernel, role and
site in the device status word, frees its tensor memory and exits; the host
reads FA_ERR_TIMEOUT; and the next normal call on the same context is
correct."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_attention_gb300 import binding
from exact_io_aware_attention_gb300 import inputs as gen
from parity import check_grad, check_lse, check_o_bf16, f64

KERNELS = {1: "forward", 3: "dK/dV", 4: "dQ", 5: "dV (d=256)", 6: "dK (d=256)", 7: "dQ (d=256)",
           8: "one-pass backward"}
ROLES = {1: "load", 2: "mma", 3: "softmax", 4: "dq"}


def decode(code):
    return (code >> 16) & 0x7FFF, (code >> 8) & 0xFF, code & 0xFF


def test_debug_configure_validates_flags():
    lib = binding.load_library()
    assert lib.fa_debug_configure(0x80, 0) == 1
    assert lib.fa_debug_configure(0, 0) == 0


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 256])
def test_stalled_producer_is_reported_and_the_context_survives(d):
    lib = binding.load_library()
    inp = gen.make_inputs(1, 2, 256, d, case=950)
    q, k, v, do = (inp[t].cuda() for t in ("q", "k", "v", "do"))
    assert binding.device_status() == 0
    try:
        assert lib.fa_debug_configure(1, 20_000_000) == 0  # 20 ms per wait
        binding.forward(q, k, v, causal=True)
        kern, role, site = decode(binding.device_status())
        assert kern == 1 and role in (2, 3), (kern, role, site)
        o0 = torch.zeros_like(q)
        lse0 = torch.zeros(q.shape[:3], device="cuda")
        # both backward forms where the head dimension has both
        for algo, kernels in ((("fused", (8,)), ("split", (3, 4))) if d < 256
                              else (("split", (5, 6, 7)),)):
            binding.backward(q, k, v, o0, do, lse0, causal=True, algo=algo)
            kern, role, site = decode(binding.device_status())
            assert kern in kernels and role in (2, 3), (algo, kern, role, site)
    finally:
        lib.fa_debug_configure(0, 0)
    # the context is intact: a normal forward and backward are correct
    o, lse = binding.forward(q, k, v, causal=True)
    dq, dk, dv = binding.backward(q, k, v, o, do, lse, causal=True)
    torch.cuda.synchronize()
    assert binding.device_status() == 0
    o_ref, lse_ref = oracle.forward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), causal=True)
    check_o_bf16(f64(o), o_ref, "after timeout")
    check_lse(f64(lse), lse_ref, "after timeout")
    g = oracle.backward(*(f64(inp[t]) for t in ("q", "k", "v", "do")), causal=True)
    for name, x in (("dq", dq), ("dk", dk), ("dv", dv)):
        check_grad(f64(x), g[name], name, "after timeout")
