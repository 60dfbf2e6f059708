"""Parity of the head-dimension-256 kernels with the fp64 oracle. Forward (one
Q tile per CTA, S double-buffered in tensor memory, K and V in 128-column
halves): dense and causal, partial tiles, Nq != Nk, fp16, the split over the
keys, strided layouts. Backward (a dV kernel and a dK / dQ kernel pair, the
streamed tiles in 128-column halves): the same cases, gradients element by
element, plus sampled rows at N = 4096."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_attention_gb300 import inputs as gen
from parity import check_grad, check_lse, check_o, f64, rel_l2

pytestmark = pytest.mark.gpu


def fa():
    import exact_io_aware_attention_gb300 as m
    return m


def check_rounded_o(o, o_ref, dtype, what):
    o = np.asarray(o, np.float64)
    rounded = torch.from_numpy(o_ref).to(dtype).double().numpy()
    r, r_floor = rel_l2(o, o_ref), rel_l2(rounded, o_ref)
    excess = float(np.sqrt(max(0.0, r * r - r_floor * r_floor)))
    beyond = float((np.abs(o - o_ref) - np.abs(rounded - o_ref)).max()) if o.size else 0.0
    assert excess <= 2e-3 and beyond <= 1e-2, f"{what} O rel_l2 excess {excess:.3e} max {beyond:.3e}"


def fwd_check(B, H, Nq, Nk, causal, case, dtype=torch.bfloat16, mask=None, splits=(None,),
              layout="bhnd", what=""):
    d = 256
    inp = gen.make_inputs(B, H, Nq, d, case, with_do=False, Nk=Nk, dtype=dtype)
    mk = None if mask is None else mask.numpy()
    o_ref, lse_ref = oracle.forward(*(f64(inp[t]) for t in ("q", "k", "v")), causal=causal,
                                    block_mask=mk)

    def dev(t):
        if layout == "bhnd":
            return t.cuda()
        return t.permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3)

    q, k, v = (dev(inp[t]) for t in ("q", "k", "v"))
    m = None if mask is None else mask.cuda()
    for ns in splits:
        o32, lse32 = fa().forward(q, k, v, causal=causal, block_mask=m, o_dtype=torch.float32,
                                  num_splits=ns)
        o, lse = fa().forward(q, k, v, causal=causal, block_mask=m, num_splits=ns)
        torch.cuda.synchronize()
        assert fa().device_status() == 0
        tag = f"{what} splits={ns}"
        check_o(f64(o32), o_ref, tag)
        check_lse(f64(lse32), lse_ref, tag)
        check_rounded_o(f64(o), o_ref, dtype, tag)
        check_lse(f64(lse), lse_ref, tag)
    return o_ref, lse_ref


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [128, 384, 1000, 2049])
def test_d256_forward(N, causal):
    fwd_check(1, 2, N, N, causal, case=960 + N % 11, what=f"d=256 N={N} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_d256_forward_fp16(causal):
    fwd_check(2, 2, 700, 700, causal, case=970, dtype=torch.float16, what="d=256 fp16")


@pytest.mark.parametrize("nq,nk", [(1, 4097), (300, 1100), (1100, 300)])
def test_d256_different_lengths_and_split(nq, nk):
    fwd_check(2, 4, nq, nk, True, case=975 + nq % 7, splits=(None, 1, 3),
              what=f"d=256 Nq={nq} Nk={nk}")


def test_d256_block_mask_and_layout():
    mask = gen.block_mask(8, 0.3, seed=980, n_key_tiles=9)
    mask[4, :] = 0
    o_ref, lse_ref = fwd_check(1, 3, 1000, 1100, False, case=981, mask=mask, layout="bnhd",
                               splits=(None, 4), what="d=256 mask bnhd")
    assert np.isneginf(lse_ref[:, :, 512:640]).all()


def bwd_check(B, H, Nq, Nk, causal, case, dtype=torch.bfloat16, mask=None, layout="bhnd",
              what=""):
    """dQ, dK, dV of the head-dimension-256 backward (fa_bwd256_dv and the two
    fa_bwd256_grad instantiations) against the oracle's analytic gradients,
    every element, from the GPU's own forward O and LSE."""
    d = 256
    inp = gen.make_inputs(B, H, Nq, d, case, Nk=Nk, dtype=dtype)
    mk = None if mask is None else mask.numpy()
    g = oracle.backward(*(f64(inp[t]) for t in ("q", "k", "v", "do")), causal=causal,
                        block_mask=mk)

    def dev(t):
        if layout == "bhnd":
            return t.cuda()
        return t.permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3)

    q, k, v, do = (dev(inp[t]) for t in ("q", "k", "v", "do"))
    m = None if mask is None else mask.cuda()
    o, lse = fa().forward(q, k, v, causal=causal, block_mask=m)
    dq, dk, dv = fa().backward(q, k, v, o, do, lse, causal=causal, block_mask=m)
    torch.cuda.synchronize()
    assert fa().device_status() == 0
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        check_grad(f64(t), g[name], name, f"{what} {name}")
    return g


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [128, 384, 1000])
def test_d256_backward(N, causal):
    bwd_check(1, 2, N, N, causal, case=990 + N % 13, what=f"d=256 bwd N={N} causal={causal}")


def test_d256_backward_fp16():
    bwd_check(2, 1, 700, 700, True, case=995, dtype=torch.float16, what="d=256 bwd fp16")


@pytest.mark.parametrize("nq,nk", [(1, 1100), (300, 1100), (1100, 300)])
def test_d256_backward_different_lengths(nq, nk):
    bwd_check(1, 2, nq, nk, True, case=996 + nq % 5, what=f"d=256 bwd Nq={nq} Nk={nk}")


def test_d256_backward_block_mask_and_layout():
    # an all-zero mask row (queries that see no key: zero dQ) and an all-zero
    # mask column (keys no query sees: zero dK and dV)
    mask = gen.block_mask(8, 0.4, seed=998, n_key_tiles=9)
    mask[4, :] = 0
    mask[:, 6] = 0
    g = bwd_check(1, 3, 1000, 1100, False, case=999, mask=mask, layout="bnhd",
                  what="d=256 bwd mask bnhd")
    assert not g["dq"][:, :, 512:640].any() and not g["dk"][:, :, 768:896].any()


def test_d256_backward_many_tiles_sampled():
    """Causal N = 4096 (32 tiles per head, every ring slot reused many times):
    whole rows of dQ, dK and dV at sampled positions against the oracle."""
    B, H, N, d = 1, 2, 4096, 256
    inp = gen.make_inputs(B, H, N, d, case=1001)
    q, k, v, do = (inp[t].cuda() for t in ("q", "k", "v", "do"))
    o, lse = fa().forward(q, k, v, causal=True)
    dq, dk, dv = fa().backward(q, k, v, o, do, lse, causal=True)
    torch.cuda.synchronize()
    assert fa().device_status() == 0
    rows = np.array([0, 1, 127, 128, 1000, 2047, 2048, 3071, 4000, 4095], np.int32)
    for h in range(H):
        sl = [f64(inp[t][:, h:h + 1]) for t in ("q", "k", "v", "do")]
        g = oracle.backward(*sl, causal=True, qrows=rows, kcols=rows)
        for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
            check_grad(f64(t[0, h, rows]), g[name][0, 0], name, f"d=256 N=4096 head {h}")
