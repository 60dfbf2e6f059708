"""Parity with the fp64 oracle for fp16 inputs and for the head dimension 96.

fp16: Q, K, V, dO are N(0, 1) rounded to fp16; the tensor cores multiply in
fp16 (P and dS rounded to fp16) and accumulate in fp32, and O, dQ, dK, dV are
fp16. Head dimension 96 has its own kernel instantiations: tiles of two
64-column chunks with zero columns 96..127 read from the tensor maps, 6
K-steps and N = 96 in the MMAs, 96 columns stored. The oracle
sees the same inputs, widened exactly to fp64. Tolerances are those of the
bf16 tests (fp16 has three more mantissa bits, so the errors are smaller)."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_attention_gb300 import FAError
from exact_io_aware_attention_gb300 import inputs as gen
from parity import check_grad, check_lse, check_o, f64, rel_l2

pytestmark = pytest.mark.gpu


def fa():
    import exact_io_aware_attention_gb300 as m
    return m


def check_rounded_o(o, o_ref, dtype, what):
    """A 16-bit O against the oracle, with its own output rounding removed
    (in quadrature for rel-L2, elementwise for max-abs), as for bf16."""
    o = np.asarray(o, np.float64)
    rounded = torch.from_numpy(o_ref).to(dtype).double().numpy()
    r, r_floor = rel_l2(o, o_ref), rel_l2(rounded, o_ref)
    excess = float(np.sqrt(max(0.0, r * r - r_floor * r_floor)))
    beyond = float((np.abs(o - o_ref) - np.abs(rounded - o_ref)).max()) if o.size else 0.0
    assert excess <= 2e-3 and beyond <= 1e-2, f"{what} O rel_l2 excess {excess:.3e} max {beyond:.3e}"


def check_all(B, H, Nq, Nk, d, causal, case, dtype, layout="bhnd", num_splits=None, what=""):
    inp = gen.make_inputs(B, H, Nq, d, case, Nk=Nk, dtype=dtype)
    scale = 1.0 / np.sqrt(d)
    x = [f64(inp[t]) for t in ("q", "k", "v", "do")]
    o_ref, lse_ref = oracle.forward(*x[:3], causal=causal, scale=scale)
    g = oracle.backward(*x, causal=causal, scale=scale)

    def dev(t):
        if layout == "bhnd":
            return t.cuda()
        return t.permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3)

    q, k, v, do = (dev(inp[t]) for t in ("q", "k", "v", "do"))
    o32, lse32 = fa().forward(q, k, v, causal=causal, o_dtype=torch.float32,
                              num_splits=num_splits)
    o, lse = fa().forward(q, k, v, causal=causal, num_splits=num_splits)
    assert o.dtype == dtype
    dq, dk, dv = fa().backward(q, k, v, o, do, lse, causal=causal)
    assert dq.dtype == dk.dtype == dv.dtype == dtype
    torch.cuda.synchronize()
    assert fa().device_status() == 0
    check_o(f64(o32), o_ref, what)
    check_lse(f64(lse32), lse_ref, what)
    check_rounded_o(f64(o), o_ref, dtype, what)
    check_lse(f64(lse), lse_ref, what)
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        check_grad(f64(t), g[name], name, what)


@pytest.mark.parametrize("d", [64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [128, 1000])
def test_fp16(N, d, causal):
    check_all(1, 2, N, N, d, causal, 900 + N % 7 + d, torch.float16,
              what=f"fp16 N={N} d={d} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [256, 1000, 4097])
def test_head_dim_96_bf16(N, causal):
    check_all(1, 2, N, N, 96, causal, 910 + N % 5, torch.bfloat16,
              what=f"d=96 N={N} causal={causal}")


def test_head_dim_96_strided_and_different_lengths():
    check_all(2, 3, 300, 1100, 96, True, 920, torch.bfloat16, layout="bnhd",
              what="d=96 bnhd Nq=300 Nk=1100")
    check_all(1, 4, 129, 700, 96, False, 921, torch.float16, layout="bnhd",
              what="fp16 d=96 bnhd")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_decode_split_96_and_fp16(dtype):
    for ns in (None, 4):
        check_all(2, 4, 1, 5000, 96, True, 930, dtype, num_splits=ns,
                  what=f"decode d=96 {dtype} splits={ns}")
    check_all(1, 8, 3, 9000, 128, True, 931, torch.float16, num_splits=None,
              what="fp16 decode d=128")


def test_head_dim_96_columns_past_96_are_not_written():
    """Outputs with a row stride of 128 elements: columns 96..127 of every row
    keep their sentinel."""
    B, H, N, d = 1, 2, 300, 96
    inp = gen.make_inputs(B, H, N, d, case=940)
    q, k, v, do = (inp[t].cuda() for t in ("q", "k", "v", "do"))
    bufs = [torch.full((B, H, N, 128), 5.0, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    o, dq, dk, dv = (b[..., :96] for b in bufs)
    _, lse = fa().forward(q, k, v, causal=True, out=o)
    fa().backward(q, k, v, o, do, lse, causal=True, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert fa().device_status() == 0
    for b in bufs:
        assert (b[..., 96:] == 5.0).all()
    o_ref, _ = oracle.forward(*(f64(inp[t]) for t in ("q", "k", "v")), causal=True)
    check_rounded_o(f64(o), o_ref, torch.bfloat16, "d=96 in a 128-column buffer")


def test_mixed_element_types_are_rejected():
    q = torch.zeros(1, 1, 128, 64, dtype=torch.float16, device="cuda")
    k = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(FAError, match="UNSUPPORTED"):
        fa().forward(q, k, k)
