"""Shared helpers of the GPU parity tests: error metrics and the tolerances the
CUDA path is held to against the fp64 oracle."""
import numpy as np
import torch

# Tolerances for bf16 inputs with fp32 accumulation.
O_REL_L2 = 2e-3
O_MAX_ABS = 1e-2
LSE_MAX_ABS = 1e-3
GRAD_REL_L2 = 5e-3


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rel_l2(x, ref):
    x, ref = np.asarray(x, np.float64), np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / (den if den > 0 else 1.0))


def max_abs(x, ref):
    x, ref = np.asarray(x, np.float64), np.asarray(ref, np.float64)
    if x.size == 0:
        return 0.0
    fin = np.isfinite(ref)
    if not np.array_equal(np.isfinite(x), fin):
        return float("inf")
    same_inf = ~fin & (x == ref)
    d = np.where(fin, np.abs(x - np.where(fin, ref, 0.0)), np.where(same_inf, 0.0, np.inf))
    return float(d.max())


def bf16_round(x):
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).to(torch.float64).numpy()


def check_o(o, o_ref, what=""):
    """O in fp32: rel-L2 and max-abs gates."""
    r, m = rel_l2(o, o_ref), max_abs(o, o_ref)
    assert r <= O_REL_L2 and m <= O_MAX_ABS, f"{what} O rel_l2={r:.3e} max_abs={m:.3e}"
    return r, m


def check_o_bf16(o, o_ref, what=""):
    """O stored in bf16. Rounding the output to bf16 adds an error independent
    of the computation's; it is removed before the gates: in quadrature for
    rel-L2 (the two errors add in quadrature) and elementwise for max-abs
    (|err| - |bf16(O_ref) - O_ref|)."""
    o = np.asarray(o, np.float64)
    rounded = bf16_round(o_ref)
    r = rel_l2(o, o_ref)
    r_floor = rel_l2(rounded, o_ref)
    r_excess = float(np.sqrt(max(0.0, r * r - r_floor * r_floor)))
    excess = float((np.abs(o - o_ref) - np.abs(rounded - o_ref)).max()) if o.size else 0.0
    assert r_excess <= O_REL_L2 and excess <= O_MAX_ABS, \
        f"{what} bf16 O rel_l2={r:.3e} (floor {r_floor:.3e}, excess {r_excess:.3e}) " \
        f"max_abs beyond rounding={excess:.3e}"
    return r_excess, excess


def check_lse(lse, lse_ref, what=""):
    m = max_abs(lse, lse_ref)
    assert m <= LSE_MAX_ABS, f"{what} LSE max_abs={m:.3e}"
    return m


def check_grad(g, g_ref, name, what=""):
    r = rel_l2(g, g_ref)
    assert r <= GRAD_REL_L2, f"{what} {name} rel_l2={r:.3e}"
    return r


def assert_same_up_to_atomics(x, y, what=""):
    """Two bf16 results of the one-pass backward's dQ, whose fp32 partial sums
    are added with atomics in whatever order the CTAs reach L2: equal up to one
    bf16 ulp of the larger value, plus an absolute floor of 1e-5 of the
    tensor's largest magnitude for elements that cancel to near zero (where
    the fp32 summation order alone moves the value by more than its ulp). A
    real defect (a lost or doubled partial) moves elements by O(1) relative."""
    xf, yf = x.float(), y.float()
    floor = 1e-5 * float(yf.abs().max())
    tol = torch.maximum(xf.abs(), yf.abs()) * 2.0 ** -7 + floor
    err = (xf - yf).abs()
    bad = err > tol
    if bad.any():
        k = int(torch.argmax(err - tol))
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.numel()} elements differ beyond one ulp; worst "
            f"{float(xf.flatten()[k]):.6e} vs {float(yf.flatten()[k]):.6e}")
