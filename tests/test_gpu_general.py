"""Parity of the CUDA path with the fp64 oracle on general shapes, through the
C ABI's strided entry points (fa_forward_ex / fa_backward_ex):

  * sequence lengths that are not a multiple of the 128-row tile (the last Q
    and K/V tiles are partial: rows past the end arrive as zeros from the
    tensor maps and must neither contribute nor be written);
  * query and key sequences of different lengths (Nq != Nk), causal masks
    aligned at the last key;
  * the [B, N, H, d] memory layout and other strided views;
  * block masks on partial tiles.

Every output element is compared with the oracle (forward O in fp32 and
bf16, LSE, dQ, dK, dV), at the tolerances of the other parity tests."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_attention_gb300 import inputs as gen
from parity import check_grad, check_lse, check_o, check_o_bf16, f64

pytestmark = pytest.mark.gpu


def fa():
    import exact_io_aware_attention_gb300 as m
    return m


def to_device(t, layout):
    """CPU [B, H, N, d] tensor -> CUDA view of the same shape, stored as
    ``layout`` ("bhnd": contiguous; "bnhd": [B, N, H, d] memory)."""
    if layout == "bhnd":
        return t.cuda()
    return t.permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3)


def run(inp, causal, scale, mask, layout="bhnd"):
    q, k, v, do = (to_device(inp[t], layout) for t in ("q", "k", "v", "do"))
    m = mask.cuda() if mask is not None else None
    o32, lse32 = fa().forward(q, k, v, causal=causal, scale=scale, block_mask=m,
                              o_dtype=torch.float32)
    o, lse = fa().forward(q, k, v, causal=causal, scale=scale, block_mask=m)
    assert o.stride() == q.stride()  # the output takes the queries' layout
    dq, dk, dv = fa().backward(q, k, v, o, do, lse, causal=causal, scale=scale, block_mask=m)
    assert dq.stride() == q.stride() and dk.stride() == k.stride()
    torch.cuda.synchronize()
    assert fa().device_status() == 0
    return o32, lse32, o, lse, dq, dk, dv


def check_all(B, H, Nq, Nk, d, causal, case, mask=None, layout="bhnd", scale=None, what=""):
    inp = gen.make_inputs(B, H, Nq, d, case, Nk=Nk)
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    mk = None if mask is None else mask.numpy()
    x = [f64(inp[t]) for t in ("q", "k", "v", "do")]
    o_ref, lse_ref = oracle.forward(*x[:3], causal=causal, scale=scale, block_mask=mk)
    g = oracle.backward(*x, causal=causal, scale=scale, block_mask=mk)
    o32, lse32, o, lse, dq, dk, dv = run(inp, causal, scale, mask, layout)
    check_o(f64(o32), o_ref, what)
    check_lse(f64(lse32), lse_ref, what)
    check_o_bf16(f64(o), o_ref, what)
    check_lse(f64(lse), lse_ref, what)
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        check_grad(f64(t), g[name], name, what)
    return o_ref, lse_ref, g, [f64(t) for t in (o, lse, dq, dk, dv)]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 129, 1000])
def test_ragged_lengths(N, d, causal):
    check_all(1, 2, N, N, d, causal, case=600 + N + d, what=f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("d,causal", [(128, True), (64, False)])
def test_ragged_length_4097(d, causal):
    """One row past 32 whole tiles: the last tile holds a single row."""
    check_all(1, 2, 4097, 4097, d, causal, case=610 + d, what=f"N=4097 d={d}")


@pytest.mark.parametrize("nq,nk,causal,d", [
    (1, 4097, True, 128),      # one new token against a long cache
    (1, 300, False, 64),
    (300, 1000, True, 64),     # prefill of 300 tokens after 700 cached ones
    (300, 1000, False, 128),
    (129, 128, True, 128),     # one query more than keys: query 0 sees nothing
    (1000, 300, True, 64),     # queries 0..699 see nothing
    (1000, 300, False, 128),
])
def test_different_query_and_key_lengths(nq, nk, causal, d):
    o_ref, lse_ref, g, (o, lse, dq, _, _) = check_all(
        1, 2, nq, nk, d, causal, case=620 + nq % 97 + nk % 89 + d,
        what=f"Nq={nq} Nk={nk} causal={causal} d={d}")
    if causal and nq > nk:
        e = nq - nk
        assert (o[:, :, :e] == 0).all() and np.isneginf(lse[:, :, :e]).all()
        assert (dq[:, :, :e] == 0).all()


@pytest.mark.parametrize("nq,nk,causal", [(1000, 1000, True), (257, 700, True), (640, 640, False)])
def test_bnhd_layout(nq, nk, causal):
    """[B, N, H, d] memory viewed as [B, H, N, d]: row stride H*d, head stride d."""
    check_all(2, 3, nq, nk, 128, causal, case=640 + nq % 7, layout="bnhd",
              what=f"bnhd Nq={nq} Nk={nk}")


@pytest.mark.parametrize("causal", [False, True])
def test_block_mask_on_partial_tiles(causal):
    nq, nk = 1000, 1100
    tq, tk = -(-nq // 128), -(-nk // 128)
    mask = gen.block_mask(tq, 0.3, seed=650 + causal, n_key_tiles=tk)
    mask[:, tk - 1] = 1       # the partial key tile, seen by every query tile
    mask[2, :] = 0            # a query tile that sees nothing
    o_ref, lse_ref, g, (o, lse, dq, _, _) = check_all(
        1, 2, nq, nk, 64, causal, case=651, mask=mask, what=f"mask causal={causal}")
    assert (o[:, :, 256:384] == 0).all() and np.isneginf(lse[:, :, 256:384]).all()
    assert (dq[:, :, 256:384] == 0).all()


def _padded(t, extra, fill):
    """CUDA view of CPU [B, H, N, d] tensor t whose storage continues past N
    with `extra` rows of `fill` in every head."""
    B, H, N, d = t.shape
    buf = torch.full((B, H, N + extra, d), fill, dtype=t.dtype, device="cuda")
    buf[:, :, :N] = t.cuda()
    return buf, buf[:, :, :N]


@pytest.mark.parametrize("nq,nk,d", [(200, 333, 64), (129, 129, 128)])
def test_rows_past_the_end_are_neither_read_nor_written(nq, nk, d):
    """Inputs whose storage continues with NaN rows after the last row of each
    head, and outputs whose storage continues with sentinel rows: the results
    match the oracle (no NaN read) and the sentinels survive (no row written
    past the end). The head stride is then (N + 136) * d, not N * d."""
    inp = gen.make_inputs(1, 3, nq, d, case=660 + d, Nk=nk)
    x = [f64(inp[t]) for t in ("q", "k", "v", "do")]
    o_ref, lse_ref = oracle.forward(*x[:3], causal=True)
    g = oracle.backward(*x, causal=True)
    nan = float("nan")
    (_, q), (_, k), (_, v), (_, do) = (_padded(inp[t], 136, nan) for t in ("q", "k", "v", "do"))
    sentinel = 7.0
    ob, o = _padded(torch.zeros(1, 3, nq, d, dtype=torch.bfloat16), 136, sentinel)
    qb, dq = _padded(torch.zeros(1, 3, nq, d, dtype=torch.bfloat16), 136, sentinel)
    kb, dk = _padded(torch.zeros(1, 3, nk, d, dtype=torch.bfloat16), 136, sentinel)
    vb, dv = _padded(torch.zeros(1, 3, nk, d, dtype=torch.bfloat16), 136, sentinel)
    _, lse = fa().forward(q, k, v, causal=True, out=o)
    fa().backward(q, k, v, o, do, lse, causal=True, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert fa().device_status() == 0
    check_o_bf16(f64(o), o_ref, "padded")
    check_lse(f64(lse), lse_ref, "padded")
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        check_grad(f64(t), g[name], name, "padded")
    for buf, n in ((ob, nq), (qb, nq), (kb, nk), (vb, nk)):
        assert (buf[:, :, n:] == sentinel).all()


def test_autograd_through_strided_views():
    """The autograd wrapper on [B, N, H, d] views returns gradients of the same
    layout and values as the oracle's."""
    B, N, H, d = 2, 333, 4, 64
    inp = gen.make_inputs(B, H, N, d, case=670)
    x = [f64(inp[t]) for t in ("q", "k", "v", "do")]
    g = oracle.backward(*x, causal=True)
    leaves = [to_device(inp[t], "bnhd").detach().requires_grad_(True) for t in ("q", "k", "v")]
    o = fa().attention(*leaves, causal=True)
    o.backward(to_device(inp["do"], "bnhd"))
    for name, leaf in zip(("dq", "dk", "dv"), leaves):
        assert leaf.grad.stride() == leaf.stride()
        check_grad(f64(leaf.grad), g[name], name, "autograd bnhd")


def test_sampled_rows_at_a_ragged_benchmark_size():
    """B=4, H=16, N=4000, d=128, causal (the medium workload with a partial
    last tile): O and LSE on sampled query rows, dK and dV on sampled key
    rows, dQ on sampled query rows, each from the oracle one by one."""
    B, H, N, d = 4, 16, 4000, 128
    inp = gen.make_inputs(B, H, N, d, case=680)
    q, k, v, do = (inp[t].cuda() for t in ("q", "k", "v", "do"))
    o, lse = fa().forward(q, k, v, causal=True)
    dq, dk, dv = fa().backward(q, k, v, o, do, lse, causal=True)
    torch.cuda.synchronize()
    assert fa().device_status() == 0
    rows = np.array([0, 1, 127, 128, 2047, 3839, 3840, 3968, 3998, 3999], np.int32)
    for b, h in ((0, 0), (3, 15)):
        sl = [f64(inp[t][b:b + 1, h:h + 1]) for t in ("q", "k", "v", "do")]
        o_ref, lse_ref = oracle.forward(*sl[:3], causal=True, rows=rows)
        g = oracle.backward(*sl, causal=True, qrows=rows, kcols=rows)
        check_o_bf16(f64(o[b, h, rows]), o_ref[0, 0], "N=4000 rows")
        check_lse(f64(lse[b, h, rows]), lse_ref[0, 0], "N=4000 rows")
        for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
            check_grad(f64(t[b, h, rows]), g[name][0, 0], name, "N=4000 rows")
