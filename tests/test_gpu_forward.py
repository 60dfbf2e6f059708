"""Parity of the CUDA forward pass (through the C ABI) with the fp64 oracle.

Small shapes are compared element by element on every output; the full-size
workloads are compared on sampled query rows, which the oracle computes one
by one (forward rows are independent)."""
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


def run_forward(inp, causal, scale, mask, o_dtype=torch.bfloat16):
    q, k, v = (inp[t].cuda() for t in ("q", "k", "v"))
    m = mask.cuda() if mask is not None else None
    o, lse = fa().forward(q, k, v, causal=causal, scale=scale, block_mask=m, o_dtype=o_dtype)
    torch.cuda.synchronize()
    assert fa().device_status() == 0
    return o, lse


def full_check(B, H, N, d, causal, case, mask=None, scale=None, what=""):
    inp = gen.make_inputs(B, H, N, d, case, with_do=False)
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    o_ref, lse_ref = oracle.forward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), causal=causal,
                                    scale=scale, block_mask=None if mask is None else mask.numpy())
    o32, lse32 = run_forward(inp, causal, scale, mask, torch.float32)
    check_o(f64(o32), o_ref, what)
    check_lse(f64(lse32), lse_ref, what)
    o16, lse16 = run_forward(inp, causal, scale, mask, torch.bfloat16)
    check_o_bf16(f64(o16), o_ref, what)
    check_lse(f64(lse16), lse_ref, what)
    return o_ref, lse_ref, f64(o16), f64(lse16)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [128, 256, 384, 640])
def test_forward_small_shapes(N, d, causal):
    full_check(1, 2, N, d, causal, case=100 + N + d, what=f"N={N} d={d} causal={causal}")


@pytest.mark.parametrize("q_tiles", ["1", "2"])
@pytest.mark.parametrize("causal,sparse", [(False, False), (True, False), (False, True)])
def test_forward_d64_q_tiles_per_cta(q_tiles, causal, sparse, monkeypatch):
    """Both d = 64 forms (one or two Q tiles per CTA, FA_FWD_Q_TILES) against the
    oracle, with a partial last tile and an odd tile count (a pair with one tile)."""
    monkeypatch.setenv("FA_FWD_Q_TILES", q_tiles)
    N = 5 * 128 - 37
    mask = gen.block_mask((N + 127) // 128, 0.5, seed=907) if sparse else None
    full_check(1, 3, N, 64, causal, case=910 + int(q_tiles), mask=mask,
               what=f"q_tiles={q_tiles} causal={causal} sparse={sparse}")


def test_forward_single_head_n256_d64():
    """The single-head workload B=1, H=1, N=256, d=64, non-causal, checked in full."""
    w = gen.WORKLOADS["single_head_n256_d64"]
    full_check(w.B, w.H, w.N, w.d, w.causal, case=w.case, what=w.name)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_forward_block_sparse_small(causal, d):
    N = 1024
    T = N // 128
    mask = gen.block_mask(T, 0.25, seed=777 + d)
    mask[3, :] = 0            # a tile row with no visible key: O = 0, LSE = -inf
    mask[5, :] = 1            # a fully dense tile row
    o_ref, lse_ref, o, lse = full_check(2, 2, N, d, causal, case=200 + d, mask=mask,
                                        what=f"sparse d={d} causal={causal}")
    assert (o[:, :, 384:512] == 0).all() and np.isneginf(lse[:, :, 384:512]).all()


@pytest.mark.parametrize("d", [64, 256])
def test_forward_scale_and_large_scores(d):
    """Scores far larger than exp's range (scale 1, |q|,|k| ~ 4): the running
    max must keep everything finite; rescales happen on many tiles. d = 256
    runs its own kernel, with its own softmax and rescale."""
    inp = gen.make_inputs(1, 2, 1024, d, case=300, with_do=False)
    for t in ("q", "k"):
        inp[t] = (inp[t].float() * 4).to(torch.bfloat16)
    o_ref, lse_ref = oracle.forward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), scale=1.0)
    o, lse = run_forward(inp, False, 1.0, None, torch.float32)
    check_o(f64(o), o_ref, "large scores")
    # LSE ~ hundreds (thousands at d = 256) here; the bound is ~1e-5 relative
    # of the fp32 scores
    assert np.abs(f64(lse) - lse_ref).max() <= 1e-3 * max(1.0, np.abs(lse_ref).max() / 64)


@pytest.mark.parametrize("d", [64, 256])
def test_forward_increasing_scores_force_rescale(d):
    """Keys whose scores grow along the sequence: the row max rises on every
    tile, so the O accumulator is rescaled repeatedly."""
    N = 1024
    inp = gen.make_inputs(1, 1, N, d, case=301, with_do=False)
    q = torch.zeros(1, 1, N, d)
    q[..., 0] = 1.0
    k = inp["k"].float()
    k[..., 0] = torch.linspace(0, 60, N)
    inp["q"], inp["k"] = q.to(torch.bfloat16), k.to(torch.bfloat16)
    for causal in (False, True):
        o_ref, lse_ref = oracle.forward(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]),
                                        causal=causal, scale=1.0)
        o, lse = run_forward(inp, causal, 1.0, None, torch.float32)
        check_o(f64(o), o_ref, f"rescale d={d} causal={causal}")
        check_lse(f64(lse), lse_ref, f"rescale d={d} causal={causal}")


def test_forward_is_deterministic():
    inp = gen.make_inputs(2, 3, 1024, 128, case=302, with_do=False)
    a = run_forward(inp, True, None, None)
    b = run_forward(inp, True, None, None)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_forward_empty_is_noop():
    q = torch.empty(2, 3, 0, 64, dtype=torch.bfloat16, device="cuda")
    o, lse = fa().forward(q, q, q)
    assert o.shape == (2, 3, 0, 64) and lse.shape == (2, 3, 0)


@pytest.mark.parametrize("name", ["gpt2_small_causal", "gpt2_medium_causal", "gpt2_medium_dense",
                                  "block_sparse_n8192"])
def test_forward_full_size_whole_heads(name):
    """Full-size workloads in the benchmark's launch configuration; the oracle
    computes every row of three heads."""
    w = gen.WORKLOADS[name]
    inp = gen.make_workload_inputs(w, with_do=False)
    mask = inp["mask"]
    o, lse = run_forward(inp, w.causal, w.scale, mask, torch.bfloat16)
    o32, lse32 = run_forward(inp, w.causal, w.scale, mask, torch.float32)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    for b, h in [(0, 0), (w.B - 1, w.H - 1), (w.B // 2, w.H // 2)]:
        sl = lambda t: f64(t[b:b + 1, h:h + 1])
        o_ref, lse_ref = oracle.forward(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), causal=w.causal,
                                        scale=w.scale,
                                        block_mask=None if mask is None else mask.numpy())
        what = f"{name} b={b} h={h}"
        check_o(f64(o32[b, h]), o_ref[0, 0], what)
        check_lse(f64(lse32[b, h]), lse_ref[0, 0], what)
        check_o_bf16(f64(o[b, h]), o_ref[0, 0], what)
        check_lse(f64(lse[b, h]), lse_ref[0, 0], what)


def test_forward_long_context_sampled_rows():
    """B=1, H=16, N=65536, d=128, causal: forward rows are independent, so the
    oracle computes uniformly drawn rows plus the tile-boundary rows of three
    heads one by one."""
    w = gen.WORKLOADS["long_context_n65536"]
    inp = gen.make_workload_inputs(w, with_do=False)
    o, lse = run_forward(inp, True, w.scale, None, torch.bfloat16)
    o32, lse32 = run_forward(inp, True, w.scale, None, torch.float32)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    rng = np.random.default_rng(w.case)
    rows = np.unique(np.concatenate([rng.choice(w.N, 64, replace=False),
                                     [0, 1, 2, 127, 128, 129, w.N - 1]])).astype(np.int32)
    for h in (0, 7, 15):
        sl = lambda t: f64(t[0:1, h:h + 1])
        o_ref, lse_ref = oracle.forward(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), causal=True,
                                        scale=w.scale, rows=rows)
        what = f"long h={h}"
        check_o(f64(o32[0, h, rows]), o_ref[0, 0], what)
        check_lse(f64(lse32[0, h, rows]), lse_ref[0, 0], what)
        check_o_bf16(f64(o[0, h, rows]), o_ref[0, 0], what)
        check_lse(f64(lse[0, h, rows]), lse_ref[0, 0], what)
