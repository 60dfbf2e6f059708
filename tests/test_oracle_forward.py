"""Pins of the fp64 oracle's forward pass against what the pages and the
mathematics fix: the printed worked examples, closed forms, invariants, brute
force on tiny inputs and the agreement of the online-softmax recurrence with
the one-shot definition."""
import math

import numpy as np
import pytest

import oracle


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _as4(x):
    x = np.asarray(x, np.float64)
    return x.reshape((1, 1) + x.shape)


# -- worked examples printed on the pages -------------------------------------

def test_worked_example_printed_values(golden):
    """p1 "Worked Example": N=2, d=2, no score scale; P rows and O printed to 3 dp."""
    g = golden("worked_example_n2_d2.txt")
    q, k, v = _as4(g["Q"]), _as4(g["K"]), _as4(g["V"])
    o, lse = oracle.forward(q, k, v, scale=g["scale"])
    tol = 0.5 * 10 ** -int(g["printed_decimals"])
    np.testing.assert_allclose(o[0, 0], np.array(g["O"]), atol=tol, rtol=0)
    # V is the identity, so O = P here: the printed P must match as well
    np.testing.assert_allclose(o[0, 0], np.array(g["P"]), atol=tol, rtol=0)
    # row 0: m = 3 and l = 1.135 as printed, so LSE = m + ln l
    assert abs(lse[0, 0, 0] - (g["row0_m"] + math.log(g["row0_l"]))) < tol / g["row0_l"] + 1e-12


def test_worked_example_closed_form():
    """Same example, exact: P = [1/(1+e^2), e^2/(1+e^2)] per row, LSE_i = max_i + ln(1+e^-2)."""
    q = _as4([[1, 0], [0, 1]])
    k = _as4([[1, 2], [3, 4]])
    v = _as4([[1, 0], [0, 1]])
    o, lse = oracle.forward(q, k, v, scale=1.0)
    e2 = math.exp(2.0)
    p = np.array([1 / (1 + e2), e2 / (1 + e2)])
    np.testing.assert_allclose(o[0, 0], np.stack([p, p]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[0, 0], [3 + math.log1p(math.exp(-2)), 4 + math.log1p(math.exp(-2))],
                               rtol=0, atol=1e-14)


def test_two_block_online_softmax_printed_values(golden):
    """p3 "A tiny worked example": blocks [1,3] then [2,5] give l = 1.203, as one-shot."""
    g = golden("two_block_online_softmax.txt")
    tol = 0.5 * 10 ** -int(g["printed_decimals"])
    scores = np.array(g["block_A"] + g["block_B"])
    n = scores.size
    q = np.ones((1, 1, n, 1))            # every query row sees the same four scores
    k = scores.reshape(1, 1, n, 1)
    v = np.ones((1, 1, n, 1))
    # block A alone
    _, lse_a = oracle.forward_tiled(q[:, :, :2], k[:, :, :2], v[:, :, :2], scale=1.0, bq=1, bk=2)
    l_a = math.exp(lse_a[0, 0, 0] - g["m_after_A"])
    assert abs(l_a - g["l_after_A"]) < tol
    # both blocks streamed through the recurrence, block size 2
    _, lse_t = oracle.forward_tiled(q, k, v, scale=1.0, bq=1, bk=2)
    l_t = math.exp(lse_t[0, 0, 0] - g["m_after_B"])
    assert abs(l_t - g["l_final"]) < tol
    assert abs(math.exp(g["m_after_A"] - g["m_after_B"]) - g["rescale_old"]) < tol
    assert abs(l_t - g["rescale_old"] * g["l_after_A"] - g["block_B_sum"]) < 2 * tol
    # and the one-shot definition agrees to rounding
    _, lse_n = oracle.forward(q, k, v, scale=1.0)
    assert abs(math.exp(lse_n[0, 0, 0] - g["m_after_B"]) - g["l_one_shot"]) < tol
    assert abs(lse_t[0, 0, 0] - lse_n[0, 0, 0]) < 1e-14
    # exact values: l = e^-4 + e^-2 + e^-3 + 1
    assert abs(l_t - (math.exp(-4) + math.exp(-2) + math.exp(-3) + 1.0)) < 1e-14


# -- closed forms and invariants ----------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_identity_values_give_p_rows_summing_to_one(causal):
    """With V = I (d = N), O is P itself: rows sum to 1, entries are non-negative,
    hidden keys get 0, and P_ij = exp(s_ij - LSE_i)."""
    n = 12
    q, k = _rand((1, 2, n, n), 1), _rand((1, 2, n, n), 2)
    v = np.broadcast_to(np.eye(n), (1, 2, n, n)).copy()
    scale = 0.37
    p, lse = oracle.forward(q, k, v, causal=causal, scale=scale)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-14)
    assert (p >= 0).all()
    s = scale * np.einsum("bhic,bhjc->bhij", q, k)
    expect = np.exp(s - lse[..., None])
    if causal:
        expect = np.where(np.tril(np.ones((n, n), bool)), expect, 0.0)
    np.testing.assert_allclose(p, expect, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_mean_of_visible_values(causal):
    """Q = 0: every visible score is 0, so O_i is the mean of V over J(i) and
    LSE_i = ln |J(i)| (|J(i)| = i + 1 when causal)."""
    n, d = 37, 5
    q = np.zeros((2, 1, n, d))
    k, v = _rand((2, 1, n, d), 3), _rand((2, 1, n, d), 4)
    o, lse = oracle.forward(q, k, v, causal=causal, scale=0.5)
    if causal:
        cnt = np.arange(1, n + 1)
        mean = np.cumsum(v, axis=2) / cnt[:, None]
    else:
        cnt = np.full(n, n)
        mean = np.broadcast_to(v.mean(axis=2, keepdims=True), v.shape)
    np.testing.assert_allclose(o, mean, rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(cnt), lse.shape), rtol=0, atol=1e-14)


def test_constant_values_give_that_constant():
    n, d = 29, 6
    q, k = _rand((1, 3, n, d), 5, 3.0), _rand((1, 3, n, d), 6, 3.0)
    c = _rand((1, 3, 1, d), 7)
    v = np.broadcast_to(c, (1, 3, n, d)).copy()
    for causal in (False, True):
        o, _ = oracle.forward(q, k, v, causal=causal)
        np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=0, atol=1e-13)


def test_shift_invariance():
    """aicassindra page, "Online softmax": adding one constant to every score of a
    row leaves softmax unchanged. With Q[..., 0] = a and K -> K + t e_0 each score
    of the row moves by scale*a*t: O is unchanged and LSE moves by scale*a*t."""
    n, d, a, t, scale = 40, 8, 1.5, 2.25, 0.3
    q, k, v = _rand((1, 2, n, d), 8), _rand((1, 2, n, d), 9), _rand((1, 2, n, d), 10)
    q[..., 0] = a
    k2 = k.copy()
    k2[..., 0] += t
    for causal in (False, True):
        o1, l1 = oracle.forward(q, k, v, causal=causal, scale=scale)
        o2, l2 = oracle.forward(q, k2, v, causal=causal, scale=scale)
        np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-13)
        np.testing.assert_allclose(l2 - l1, scale * a * t, rtol=0, atol=1e-12)


def test_key_permutation_equivariance():
    """Non-causal, no mask: permuting keys and values together leaves O alone;
    permuting queries permutes the rows of O and LSE."""
    n, d = 33, 7
    q, k, v = _rand((1, 1, n, d), 11), _rand((1, 1, n, d), 12), _rand((1, 1, n, d), 13)
    perm = np.random.default_rng(14).permutation(n)
    o, lse = oracle.forward(q, k, v)
    o2, lse2 = oracle.forward(q, k[:, :, perm], v[:, :, perm])
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-14)
    o3, lse3 = oracle.forward(q[:, :, perm], k, v)
    np.testing.assert_allclose(o3, o[:, :, perm], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse3, lse[:, :, perm], rtol=0, atol=1e-15)


def test_single_key_row_copies_value():
    """Causal row 0 sees only key 0: O_0 = V_0 exactly and LSE_0 = s_00."""
    n, d = 9, 4
    q, k, v = _rand((1, 1, n, d), 15), _rand((1, 1, n, d), 16), _rand((1, 1, n, d), 17)
    o, lse = oracle.forward(q, k, v, causal=True, scale=0.7)
    np.testing.assert_array_equal(o[0, 0, 0], v[0, 0, 0])
    assert abs(lse[0, 0, 0] - 0.7 * float(q[0, 0, 0] @ k[0, 0, 0])) < 1e-15


# -- masks: brute force from an explicit N x N visibility matrix ---------------

def _visible(n, causal, mask, tile):
    vis = np.ones((n, n), bool)
    for i in range(n):
        for j in range(n):
            if causal and j > i:
                vis[i, j] = False
            if mask is not None and not mask[i // tile][j // tile]:
                vis[i, j] = False
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


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,tile", [(16, 4), (22, 4), (24, 8)])
def test_block_mask_against_brute_force(causal, n, tile):
    t = (n + tile - 1) // tile
    rng = np.random.default_rng(100 + n + tile + causal)
    mask = (rng.random((t, t)) < 0.4).astype(np.uint8)
    mask[np.arange(t), np.arange(t)] = 1
    mask[1, :] = 0  # one tile row fully hidden: those rows have no visible key
    d = 5
    q, k, v = _rand((1, 2, n, d), 18), _rand((1, 2, n, d), 19), _rand((1, 2, n, d), 20)
    vis = _visible(n, causal, mask, tile)
    o_ref, lse_ref = _brute(q, k, v, 0.45, vis)
    o, lse = oracle.forward(q, k, v, causal=causal, scale=0.45, block_mask=mask, mask_tile=tile)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-13)
    hidden = slice(tile, min(2 * tile, n))
    assert (o[:, :, hidden] == 0).all() and np.isneginf(lse[:, :, hidden]).all()


def test_all_ones_mask_is_dense_and_lower_tile_mask_is_causal():
    n, tile, d = 20, 4, 3
    t = n // tile
    q, k, v = _rand((1, 1, n, d), 21), _rand((1, 1, n, d), 22), _rand((1, 1, n, d), 23)
    dense = oracle.forward(q, k, v)
    ones = oracle.forward(q, k, v, block_mask=np.ones((t, t), np.uint8), mask_tile=tile)
    for a, b in zip(dense, ones):
        np.testing.assert_array_equal(a, b)
    causal = oracle.forward(q, k, v, causal=True)
    lower = oracle.forward(q, k, v, causal=True, block_mask=np.tril(np.ones((t, t), np.uint8)),
                           mask_tile=tile)
    for a, b in zip(causal, lower):
        np.testing.assert_array_equal(a, b)


def test_row_subset_matches_full():
    n, d = 50, 6
    q, k, v = _rand((2, 2, n, d), 24), _rand((2, 2, n, d), 25), _rand((2, 2, n, d), 26)
    rows = [0, 7, 49, 13, 13]
    o, lse = oracle.forward(q, k, v, causal=True)
    o_r, lse_r = oracle.forward(q, k, v, causal=True, rows=rows)
    np.testing.assert_array_equal(o_r, o[:, :, rows])
    np.testing.assert_array_equal(lse_r, lse[:, :, rows])


def test_empty_sequence():
    z = np.zeros((1, 2, 0, 4))
    o, lse = oracle.forward(z, z, z)
    assert o.shape == (1, 2, 0, 4) and lse.shape == (1, 2, 0)


# -- the online-softmax recurrence equals the definition ----------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("bq,bk", [(64, 64), (128, 128), (7, 5), (1, 300)])
def test_tiled_recurrence_matches_definition(causal, bq, bk):
    """muhibwaqar "build it from scratch": the blocked loop equals the naive
    function to floating-point noise (here fp64: 1e-12 relative)."""
    n, d = 300, 16
    q, k, v = _rand((1, 2, n, d), 27, 2.0), _rand((1, 2, n, d), 28, 2.0), _rand((1, 2, n, d), 29)
    o, lse = oracle.forward(q, k, v, causal=causal)
    ot, lset = oracle.forward_tiled(q, k, v, causal=causal, bq=bq, bk=bk)
    assert np.linalg.norm(ot - o) <= 1e-12 * np.linalg.norm(o)
    np.testing.assert_allclose(lset, lse, rtol=1e-13, atol=0)


def test_tiled_recurrence_with_block_mask():
    n, tile, d = 48, 8, 4
    t = n // tile
    mask = (np.random.default_rng(30).random((t, t)) < 0.3).astype(np.uint8)
    mask[2, :] = 0
    q, k, v = _rand((1, 1, n, d), 31), _rand((1, 1, n, d), 32), _rand((1, 1, n, d), 33)
    for causal in (False, True):
        o, lse = oracle.forward(q, k, v, causal=causal, block_mask=mask, mask_tile=tile)
        ot, lset = oracle.forward_tiled(q, k, v, causal=causal, block_mask=mask, mask_tile=tile,
                                        bq=5, bk=3)
        np.testing.assert_allclose(ot, o, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lset, lse, rtol=1e-13, atol=0)


def test_large_scores_stay_finite():
    """Scores far beyond exp's range: the max subtraction keeps everything finite."""
    n, d = 64, 4
    q, k, v = _rand((1, 1, n, d), 34, 40.0), _rand((1, 1, n, d), 35, 40.0), _rand((1, 1, n, d), 36)
    o, lse = oracle.forward(q, k, v, scale=1.0)
    ot, lset = oracle.forward_tiled(q, k, v, scale=1.0, bq=16, bk=16)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    np.testing.assert_allclose(ot, o, rtol=1e-11, atol=1e-13)
