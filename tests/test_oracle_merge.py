"""Pins of the oracle's block merge (the rule that combines the softmax
results of disjoint key blocks, "Paper Notes: FlashAttention", section
"Tiling: Block-by-Block Softmax"): the printed two-block example, and the
merge of key blocks computed one by one against the one-shot definition."""
import math

import numpy as np
import pytest

import oracle


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def test_printed_two_block_example(golden):
    """aicassindra, "A tiny worked example": blocks [1, 3] and [2, 5]; after A
    m = 3, l = 1.135; the old sum is rescaled by e^(3-5) = 0.135; B's sum is
    1.050; the merged l = 1.203 equals the one-shot sum."""
    g = golden("two_block_online_softmax.txt")
    tol = 0.5 * 10 ** -int(g["printed_decimals"])
    a, b = np.array(g["block_A"], float), np.array(g["block_B"], float)
    stats = []
    for blk in (a, b):
        m = blk.max()
        stats.append((m, np.exp(blk - m).sum()))
    (m_a, l_a), (m_b, l_b) = stats
    assert m_a == g["m_after_A"] and abs(l_a - g["l_after_A"]) < tol
    assert abs(l_b - g["block_B_sum"]) < tol
    o_a, o_b = np.array([[1.0, 0.0]]), np.array([[0.0, 1.0]])  # any normalised outputs
    o, m, l = oracle.merge([o_a, o_b], [np.array([m_a]), np.array([m_b])],
                           [np.array([l_a]), np.array([l_b])])
    assert m[0] == g["m_after_B"]
    assert abs(math.exp(m_a - m[0]) - g["rescale_old"]) < tol
    assert abs(l[0] - g["l_final"]) < tol and abs(l[0] - g["l_one_shot"]) < tol
    # the output weights are the blocks' shares of the merged sum
    np.testing.assert_allclose(o[0], [math.exp(m_a - m_b) * l_a / l[0], l_b / l[0]], rtol=1e-15)


@pytest.mark.parametrize("cuts", [[0, 300], [0, 150, 300], [0, 50, 51, 200, 300],
                                  [0, 7, 19, 64, 127, 128, 250, 299, 300]])
def test_merge_of_key_blocks_equals_the_definition(cuts):
    """Partial (O_s, LSE_s) of each key block from the oracle's definition,
    merged, equal the definition over all keys."""
    B, H, Nq, Nk, d = 2, 3, 37, 300, 16
    q, k, v = _rand((B, H, Nq, d), 700, 1.5), _rand((B, H, Nk, d), 701, 1.5), _rand((B, H, Nk, d), 702)
    o_ref, lse_ref = oracle.forward(q, k, v, scale=0.4)
    parts = [oracle.forward(q, k[:, :, a:b], v[:, :, a:b], scale=0.4)
             for a, b in zip(cuts[:-1], cuts[1:])]
    o, lse = oracle.merge_lse([p[0] for p in parts], [p[1] for p in parts])
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-14, atol=0)
    # the order of the blocks does not matter
    order = list(reversed(range(len(parts))))
    o2, lse2 = oracle.merge_lse([parts[i][0] for i in order], [parts[i][1] for i in order])
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=1e-14, atol=0)


def test_blocks_without_keys():
    """A block in which a row sees nothing (LSE = -inf, O = 0) leaves the other
    blocks' result unchanged; a row that sees nothing anywhere gets O = 0 and
    LSE = -inf."""
    o1 = _rand((4, 8), 710)
    lse1 = _rand((4,), 711)
    empty_o, empty_lse = np.zeros((4, 8)), np.full(4, -np.inf)
    o, lse = oracle.merge_lse([empty_o, o1, empty_o], [empty_lse, lse1, empty_lse])
    np.testing.assert_allclose(o, o1, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, lse1, rtol=1e-15, atol=0)
    o, lse = oracle.merge_lse([empty_o, empty_o], [empty_lse, empty_lse])
    assert (o == 0).all() and np.isneginf(lse).all()


def test_large_score_gaps_stay_finite():
    """Block maxima hundreds apart: the rescale factors underflow to 0 for the
    small blocks and nothing overflows."""
    o_parts = [_rand((3, 4), 720 + s) for s in range(3)]
    lse_parts = [np.array([0.0, 800.0, -700.0]), np.array([900.0, 1.0, -710.0]),
                 np.array([-5.0, 2.0, -705.0])]
    o, lse = oracle.merge_lse(o_parts, lse_parts)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    np.testing.assert_allclose(o[0], o_parts[1][0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(o[1], o_parts[0][1], rtol=0, atol=1e-15)
    w = np.exp(np.array([-700.0, -710.0, -705.0]) - (-700.0))
    np.testing.assert_allclose(o[2], sum(w[s] * o_parts[s][2] for s in range(3)) / w.sum(),
                               rtol=1e-14)
