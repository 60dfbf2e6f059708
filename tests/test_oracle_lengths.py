"""Pins of the oracle for query and key sequences of different lengths
(Nq != Nk) and for lengths that are not a multiple of any tile.

The pages define causal attention for one sequence (query i sees key j iff
j <= i). For Nq != Nk the oracle aligns the last query with the last key
(j <= i + Nk - Nq): the Nq queries are the last Nq positions of a sequence
whose Nk keys are all present, as when new tokens attend to a cache. These
tests pin that reading to the pages' one-sequence rule, which the other oracle
tests pin to the printed examples: the rectangular problem must reproduce the
matching rows of the square problem, forward and backward. They also check it
against brute force over an explicit visibility matrix, against fp64 autograd
on the CPU (torch) and against central finite differences."""
import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _visible(nq, nk, causal, mask=None, tile=1):
    i = np.arange(nq)[:, None]
    j = np.arange(nk)[None, :]
    vis = np.ones((nq, nk), bool)
    if causal:
        vis &= j <= i + (nk - nq)
    if mask is not None:
        vis &= np.asarray(mask, bool)[i // tile, j // tile]
    return vis


def _brute(q, k, v, scale, vis):
    s = scale * np.einsum("bhic,bhjc->bhij", q, k)
    s = np.where(vis, s, -np.inf)
    m = s.max(-1, keepdims=True)
    empty = ~np.isfinite(m)
    e = np.where(vis, np.exp(s - np.where(empty, 0.0, m)), 0.0)
    l = e.sum(-1, keepdims=True)
    o = np.where(empty, 0.0, e / np.where(empty, 1.0, l)) @ v
    lse = np.where(empty[..., 0], -np.inf, (m + np.log(np.where(empty, 1.0, l)))[..., 0])
    return o, lse


# -- the rectangular causal rule reproduces rows of the square problem --------

@pytest.mark.parametrize("n,m", [(40, 1), (40, 13), (300, 129), (257, 256)])
def test_last_queries_reproduce_rows_of_the_full_sequence(n, m):
    """Queries = the last m positions, keys = all n: O, LSE and dQ equal rows
    n-m.. of the n x n causal problem; dK, dV equal the square problem's with
    the upstream gradient zero on the first n-m rows."""
    d = 8
    q, k, v, do = (_rand((1, 2, n, d), 400 + i) for i in range(4))
    do[:, :, : n - m] = 0.0
    o, lse = oracle.forward(q, k, v, causal=True, scale=0.3)
    g = oracle.backward(q, k, v, do, causal=True, scale=0.3)
    o_r, lse_r = oracle.forward(q[:, :, n - m:], k, v, causal=True, scale=0.3)
    g_r = oracle.backward(q[:, :, n - m:], k, v, do[:, :, n - m:], causal=True, scale=0.3)
    np.testing.assert_array_equal(o_r, o[:, :, n - m:])
    np.testing.assert_array_equal(lse_r, lse[:, :, n - m:])
    np.testing.assert_allclose(g_r["dq"], g["dq"][:, :, n - m:], rtol=0, atol=1e-14)
    np.testing.assert_allclose(g_r["dk"], g["dk"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(g_r["dv"], g["dv"], rtol=0, atol=1e-13)


def test_single_query_sees_every_key():
    """One query at the end of the sequence: causal and dense agree."""
    q, k, v = _rand((2, 3, 1, 16), 410), _rand((2, 3, 77, 16), 411), _rand((2, 3, 77, 16), 412)
    oc, lc = oracle.forward(q, k, v, causal=True)
    od, ld = oracle.forward(q, k, v, causal=False)
    np.testing.assert_array_equal(oc, od)
    np.testing.assert_array_equal(lc, ld)


@pytest.mark.parametrize("nq,nk", [(50, 20), (129, 128)])
def test_more_queries_than_keys(nq, nk):
    """Queries before the first key see nothing (O = 0, LSE = -inf); the last
    nk queries form the square causal problem over the nk keys."""
    d = 6
    q, do = _rand((1, 2, nq, d), 420), _rand((1, 2, nq, d), 421)
    k, v = _rand((1, 2, nk, d), 422), _rand((1, 2, nk, d), 423)
    o, lse = oracle.forward(q, k, v, causal=True)
    g = oracle.backward(q, k, v, do, causal=True)
    e = nq - nk
    assert (o[:, :, :e] == 0).all() and np.isneginf(lse[:, :, :e]).all()
    assert (g["dq"][:, :, :e] == 0).all()
    o_s, lse_s = oracle.forward(q[:, :, e:], k, v, causal=True)
    g_s = oracle.backward(q[:, :, e:], k, v, do[:, :, e:], causal=True)
    np.testing.assert_array_equal(o[:, :, e:], o_s)
    np.testing.assert_array_equal(lse[:, :, e:], lse_s)
    for name in ("dq",):
        np.testing.assert_allclose(g[name][:, :, e:], g_s[name], rtol=0, atol=1e-14)
    for name in ("dk", "dv"):
        np.testing.assert_allclose(g[name], g_s[name], rtol=0, atol=1e-13)


# -- brute force and independent evaluations ----------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk,tile", [(23, 41, 4), (41, 23, 4), (9, 9, 4), (1, 30, 8)])
def test_rectangular_block_mask_against_brute_force(causal, nq, nk, tile):
    tq, tk = -(-nq // tile), -(-nk // tile)
    rng = np.random.default_rng(430 + nq + nk + causal)
    mask = (rng.random((tq, tk)) < 0.6).astype(np.uint8)
    d = 5
    q, k, v = _rand((2, 1, nq, d), 431), _rand((2, 1, nk, d), 432), _rand((2, 1, nk, d), 433)
    o_ref, lse_ref = _brute(q, k, v, 0.5, _visible(nq, nk, causal, mask, tile))
    o, lse = oracle.forward(q, k, v, causal=causal, scale=0.5, block_mask=mask, mask_tile=tile)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-13)
    ot, lset = oracle.forward_tiled(q, k, v, causal=causal, scale=0.5, block_mask=mask,
                                    mask_tile=tile, bq=3, bk=5)
    np.testing.assert_allclose(ot, o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lset, lse, rtol=1e-13, atol=0)


def _torch_grads(q, k, v, do, vis, scale):
    t = [torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v)]
    s = (scale * t[0] @ t[1].transpose(-1, -2)).masked_fill(~torch.tensor(vis), float("-inf"))
    o = torch.softmax(s, dim=-1) @ t[2]
    o.backward(torch.tensor(do))
    return o.detach().numpy(), torch.logsumexp(s, -1).detach().numpy(), [x.grad.numpy() for x in t]


@pytest.mark.parametrize("nq,nk,causal", [(129, 129, True), (129, 129, False), (70, 200, True),
                                          (200, 333, False), (1, 257, True)])
def test_gradients_match_torch_autograd_fp64(nq, nk, causal):
    """Lengths that are no multiple of 128, and Nq != Nk (every query row sees
    at least one key, so torch's softmax is defined on every row)."""
    d, scale = 16, 0.25
    q, do = _rand((1, 2, nq, d), 440), _rand((1, 2, nq, d), 441)
    k, v = _rand((1, 2, nk, d), 442), _rand((1, 2, nk, d), 443)
    o_t, lse_t, (dq_t, dk_t, dv_t) = _torch_grads(q, k, v, do, _visible(nq, nk, causal), scale)
    o, lse = oracle.forward(q, k, v, causal=causal, scale=scale)
    g = oracle.backward(q, k, v, do, causal=causal, scale=scale)
    np.testing.assert_allclose(o, o_t, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_t, rtol=0, atol=1e-12)
    for a, b in ((g["dq"], dq_t), (g["dk"], dk_t), (g["dv"], dv_t)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)


def test_rectangular_gradients_match_finite_differences():
    nq, nk, d, kw = 5, 7, 3, dict(causal=True, scale=0.9)
    x = {"q": _rand((1, 1, nq, d), 450), "k": _rand((1, 1, nk, d), 451),
         "v": _rand((1, 1, nk, d), 452), "do": _rand((1, 1, nq, d), 453)}
    g = oracle.backward(x["q"], x["k"], x["v"], x["do"], **kw)

    def loss():
        return float((oracle.forward(x["q"], x["k"], x["v"], **kw)[0] * x["do"]).sum())

    h = 1e-6
    for name, key in (("q", "dq"), ("k", "dk"), ("v", "dv")):
        a = x[name]
        fd = np.zeros_like(a)
        for idx in np.ndindex(a.shape):
            orig = a[idx]
            a[idx] = orig + h
            lp = loss()
            a[idx] = orig - h
            lm = loss()
            a[idx] = orig
            fd[idx] = (lp - lm) / (2 * h)
        assert np.abs(g[key] - fd).max() <= 1e-6 * max(1.0, np.abs(fd).max()), name


def test_no_keys():
    q = _rand((1, 1, 3, 4), 460)
    z = np.zeros((1, 1, 0, 4))
    o, lse = oracle.forward(q, z, z, causal=False)
    assert (o == 0).all() and np.isneginf(lse).all()
    g = oracle.backward(q, z, z, q)
    assert (g["dq"] == 0).all() and g["dk"].shape == (1, 1, 0, 4)
