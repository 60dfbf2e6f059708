"""Parity of the forward pass with the keys split over several CTAs
(fa_forward_split_ex) with the fp64 oracle: decode and prefill shapes against
long key sequences, forced and library-chosen split counts, causal and
block-sparse masks, partial tiles, fp32 and bf16 outputs. The merged result is
compared with the oracle's definition over all keys; the merge itself is the
pages' block-merge rule, which tests/test_oracle_merge.py pins."""
import numpy as np
import pytest
import torch

import oracle
from exact_io_aware_attention_gb300 import inputs as gen
from parity import check_lse, check_o, check_o_bf16, f64

pytestmark = pytest.mark.gpu


def fa():
    import exact_io_aware_attention_gb300 as m
    return m


def split_check(B, H, Nq, Nk, d, causal, splits, case, mask=None, what=""):
    inp = gen.make_inputs(B, H, Nq, d, case, with_do=False, Nk=Nk)
    scale = 1.0 / np.sqrt(d)
    mk = None if mask is None else mask.numpy()
    o_ref, lse_ref = oracle.forward(*(f64(inp[t]) for t in ("q", "k", "v")), causal=causal,
                                    scale=scale, block_mask=mk)
    q, k, v = (inp[t].cuda() for t in ("q", "k", "v"))
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
        check_o_bf16(f64(o), o_ref, tag)
        check_lse(f64(lse), lse_ref, tag)
    return o_ref, lse_ref


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", [
    (2, 8, 1, 4097, 128, True),       # decode: one new token, 4097 cached keys
    (1, 4, 1, 65536, 64, False),      # decode against the longest supported cache
    (1, 16, 1, 65536, 128, True),
    (2, 3, 200, 3000, 128, True),     # a prefill chunk after 2800 cached tokens
    (1, 2, 129, 1000, 64, False),     # two query tiles, the second partial
])
def test_split_forward_matches_the_oracle(B, H, Nq, Nk, d, causal):
    auto = fa().default_num_splits(B, H, Nq, Nk, d, causal)
    tiles = -(-Nk // 128)
    forced = sorted({2, 3, min(16, tiles), min(128, tiles)})
    split_check(B, H, Nq, Nk, d, causal, [auto] + forced, case=800 + Nq % 13 + d,
                what=f"B={B} H={H} Nq={Nq} Nk={Nk} d={d} causal={causal}")


def test_library_splits_decode_and_not_training_shapes():
    assert fa().default_num_splits(1, 16, 1, 65536, 128, True) > 1
    assert fa().default_num_splits(2, 8, 1, 4097, 64, False) > 1
    # every SM already has a CTA: no split
    assert fa().default_num_splits(4, 16, 4096, 4096, 128, True) == 1
    # too few key tiles to share
    assert fa().default_num_splits(1, 1, 1, 300, 128, False) == 1


def test_more_splits_than_key_tiles():
    """Splits without any K/V tile write LSE = -inf partials, which the merge
    ignores."""
    split_check(1, 2, 64, 300, 128, False, [7, 16], case=810, what="empty splits")


def test_split_with_block_mask_and_empty_rows():
    nq, nk = 256, 2048
    mask = gen.block_mask(2, 0.3, seed=820, n_key_tiles=16)
    mask[1, :] = 0  # the second query tile sees nothing: O = 0, LSE = -inf
    o_ref, lse_ref = split_check(1, 3, nq, nk, 64, False, [4, 16], case=821, mask=mask,
                                 what="masked")
    assert (o_ref[:, :, 128:] == 0).all() and np.isneginf(lse_ref[:, :, 128:]).all()


def test_split_with_strided_layout():
    """[B, N, H, d] memory for every operand, and an output view into a larger
    buffer whose other rows must survive."""
    B, H, Nq, Nk, d = 2, 4, 3, 2000, 128
    inp = gen.make_inputs(B, H, Nq, d, case=830, with_do=False, Nk=Nk)
    o_ref, lse_ref = oracle.forward(*(f64(inp[t]) for t in ("q", "k", "v")), causal=True)
    q, k, v = (inp[t].permute(0, 2, 1, 3).contiguous().cuda().permute(0, 2, 1, 3)
               for t in ("q", "k", "v"))
    buf = torch.full((B, H, Nq + 5, d), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[:, :, 2:2 + Nq]
    o, lse = fa().forward(q, k, v, causal=True, out=out, num_splits=5)
    torch.cuda.synchronize()
    assert fa().device_status() == 0
    check_o_bf16(f64(o), o_ref, "strided split")
    check_lse(f64(lse), lse_ref, "strided split")
    assert (buf[:, :, :2] == 7.0).all() and (buf[:, :, 2 + Nq:] == 7.0).all()


def test_split_and_plain_forward_agree_and_backward_accepts_either():
    """The split forward's O and LSE feed the backward pass like the plain
    forward's: the gradients from both agree to rounding."""
    B, H, Nq, Nk, d = 1, 4, 64, 4096, 128
    inp = gen.make_inputs(B, H, Nq, d, case=840, Nk=Nk)
    q, k, v, do = (inp[t].cuda() for t in ("q", "k", "v", "do"))
    o1, lse1 = fa().forward(q, k, v, causal=True, num_splits=1)
    o2, lse2 = fa().forward(q, k, v, causal=True, num_splits=8)
    g1 = fa().backward(q, k, v, o1, do, lse1, causal=True)
    g2 = fa().backward(q, k, v, o2, do, lse2, causal=True)
    torch.cuda.synchronize()
    assert fa().device_status() == 0
    assert float((lse1 - lse2).abs().max()) < 1e-4
    for a, b in zip(g1, g2):
        rel = float((a.float() - b.float()).norm() / b.float().norm())
        assert rel < 5e-3, rel
