"""Pins of the fp64 oracle's gradients. The pages give no gradient formulas, so
the gradients are pinned by what the mathematics fixes: central finite
differences of L = sum(dO * O), the zero row sums of the softmax Jacobian, the
identity D_i = dO_i . O_i, and an independent fp64 autograd evaluation on the
CPU (torch), plus agreement of row/column subsets with the full computation."""
import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _loss(q, k, v, do, **kw):
    o, _ = oracle.forward(q, k, v, **kw)
    return float((o * do).sum())


def _fd_grad(x_name, inputs, kw, h=1e-6):
    base = dict(inputs)
    x = base[x_name]
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        orig = x[idx]
        x[idx] = orig + h
        lp = _loss(base["q"], base["k"], base["v"], base["do"], **kw)
        x[idx] = orig - h
        lm = _loss(base["q"], base["k"], base["v"], base["do"], **kw)
        x[idx] = orig
        g[idx] = (lp - lm) / (2 * h)
    return g


CASES = [
    dict(name="dense", n=6, d=3, kw=dict(scale=0.8)),
    dict(name="causal", n=7, d=4, kw=dict(causal=True, scale=1.3)),
    dict(name="masked", n=8, d=2, kw=dict(block_mask=np.array([[1, 0, 1, 0], [0, 1, 1, 0],
                                                               [1, 0, 0, 1], [0, 0, 0, 0]],
                                                              np.uint8), mask_tile=2, scale=0.6)),
    dict(name="causal_masked", n=8, d=3, kw=dict(causal=True, block_mask=np.array(
        [[1, 1, 0, 1], [1, 0, 1, 1], [0, 1, 1, 0], [1, 1, 0, 1]], np.uint8), mask_tile=2)),
]


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_gradients_match_finite_differences(case):
    n, d, kw = case["n"], case["d"], case["kw"]
    inputs = {t: _rand((1, 2, n, d), 40 + i) for i, t in enumerate(("q", "k", "v", "do"))}
    g = oracle.backward(inputs["q"], inputs["k"], inputs["v"], inputs["do"], **kw)
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv")):
        fd = _fd_grad(name, {t: a.copy() for t, a in inputs.items()}, kw)
        err = np.abs(g[key] - fd).max()
        assert err <= 1e-6 * max(1.0, np.abs(fd).max()), (name, err)


def _torch_reference(q, k, v, do, causal, scale, vis=None):
    t = [torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v)]
    s = scale * t[0] @ t[1].transpose(-1, -2)
    n = q.shape[-2]
    allowed = torch.ones(n, n, dtype=torch.bool)
    if causal:
        allowed &= torch.tril(torch.ones(n, n, dtype=torch.bool))
    if vis is not None:
        allowed &= torch.tensor(vis)
    s = s.masked_fill(~allowed, float("-inf"))
    o = torch.softmax(s, dim=-1) @ t[2]
    lse = torch.logsumexp(s, dim=-1)
    o.backward(torch.tensor(do))
    return o.detach().numpy(), lse.detach().numpy(), [x.grad.numpy() for x in t]


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_torch_autograd_fp64(causal):
    """Independent library evaluation (torch softmax + autograd, fp64, CPU)."""
    n, d, scale = 150, 24, 1 / np.sqrt(24)
    q, k, v, do = (_rand((2, 3, n, d), 50 + i) for i in range(4))
    o_t, lse_t, (dq_t, dk_t, dv_t) = _torch_reference(q, k, v, do, causal, scale)
    o, lse = oracle.forward(q, k, v, causal=causal, scale=scale)
    g = oracle.backward(q, k, v, do, causal=causal, scale=scale)
    np.testing.assert_allclose(o, o_t, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_t, rtol=0, atol=1e-12)
    np.testing.assert_allclose(g["lse"], lse_t, rtol=0, atol=1e-12)
    for a, b in ((g["dq"], dq_t), (g["dk"], dk_t), (g["dv"], dv_t)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)


def test_block_mask_gradients_match_torch_autograd_fp64():
    n, tile, d = 64, 16, 8
    t = n // tile
    mask = (np.random.default_rng(60).random((t, t)) < 0.5).astype(np.uint8)
    mask[np.arange(t), np.arange(t)] = 1
    vis = np.kron(mask, np.ones((tile, tile), np.uint8)).astype(bool)
    q, k, v, do = (_rand((1, 2, n, d), 61 + i) for i in range(4))
    _, _, (dq_t, dk_t, dv_t) = _torch_reference(q, k, v, do, False, 0.35, vis)
    g = oracle.backward(q, k, v, do, scale=0.35, block_mask=mask, mask_tile=tile)
    for a, b in ((g["dq"], dq_t), (g["dk"], dk_t), (g["dv"], dv_t)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_softmax_jacobian_and_row_statistics(causal):
    """sum_j dS_ij = 0 for every row, hence sum_j dK_j = 0 per head; and
    D_i = sum_j P_ij dP_ij equals dO_i . O_i; LSE agrees with the forward."""
    n, d = 90, 12
    q, k, v, do = (_rand((2, 2, n, d), 70 + i) for i in range(4))
    g = oracle.backward(q, k, v, do, causal=causal)
    o, lse = oracle.forward(q, k, v, causal=causal)
    np.testing.assert_allclose(g["dk"].sum(axis=2), 0.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(g["D"], (do * o).sum(-1), rtol=0, atol=1e-12)
    np.testing.assert_allclose(g["lse"], lse, rtol=0, atol=1e-13)


def test_constant_values_give_zero_query_and_key_gradients():
    """V constant over keys makes O independent of Q and K: dQ = dK = 0 and
    dV_j = sum_i P_ij dO_i sums to sum_i dO_i over keys."""
    n, d = 40, 6
    q, k, do = _rand((1, 2, n, d), 80), _rand((1, 2, n, d), 81), _rand((1, 2, n, d), 82)
    v = np.broadcast_to(_rand((1, 2, 1, d), 83), (1, 2, n, d)).copy()
    g = oracle.backward(q, k, v, do, causal=True)
    np.testing.assert_allclose(g["dq"], 0.0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(g["dk"], 0.0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(g["dv"].sum(axis=2), do.sum(axis=2), rtol=0, atol=1e-12)


def test_subsets_match_full():
    n, d = 70, 5
    q, k, v, do = (_rand((1, 3, n, d), 90 + i) for i in range(4))
    full = oracle.backward(q, k, v, do, causal=True)
    rows, cols = [3, 69, 0, 35], [69, 1, 0, 44, 44]
    part = oracle.backward(q, k, v, do, causal=True, qrows=rows, kcols=cols)
    np.testing.assert_array_equal(part["dq"], full["dq"][:, :, rows])
    np.testing.assert_array_equal(part["dk"], full["dk"][:, :, cols])
    np.testing.assert_array_equal(part["dv"], full["dv"][:, :, cols])
    only_q = oracle.backward(q, k, v, do, causal=True, want_dkv=False)
    np.testing.assert_array_equal(only_q["dq"], full["dq"])
    assert only_q["dk"].shape[2] == 0


def test_hidden_rows_and_keys_get_zero_gradient():
    """A tile row of the mask that is all zero: those queries see nothing, so
    their dQ is 0; a key column that is all zero gets dK = dV = 0."""
    n, tile, d = 12, 4, 3
    mask = np.array([[1, 0, 1], [0, 0, 0], [1, 0, 1]], np.uint8)
    q, k, v, do = (_rand((1, 1, n, d), 95 + i) for i in range(4))
    g = oracle.backward(q, k, v, do, block_mask=mask, mask_tile=tile)
    assert (g["dq"][:, :, 4:8] == 0).all()
    assert (g["dk"][:, :, 4:8] == 0).all() and (g["dv"][:, :, 4:8] == 0).all()
    assert np.isneginf(g["lse"][:, :, 4:8]).all()
