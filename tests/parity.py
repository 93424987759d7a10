"""Tolerance check shared by the GPU parity tests.

The bar: |got - ref| <= 2e-5 + 1e-6 * |ref| element by element against the
oracle's float64 result; NaN must meet NaN and +-inf the same infinity.
"""
import numpy as np

TOL_ABS = 2e-5
TOL_REL = 1e-6


def assert_parity(got, ref, what=""):
    if hasattr(got, "detach"):
        got = got.detach().cpu().numpy()
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    nan_g, nan_r = np.isnan(got), np.isnan(ref)
    assert np.array_equal(nan_g, nan_r), (
        f"{what}: NaN mismatch at {np.argwhere(nan_g != nan_r)[:5].tolist()}")
    inf_r = np.isinf(ref)
    assert np.array_equal(got[inf_r], ref[inf_r]) and not np.isinf(got[~inf_r]).any(), (
        f"{what}: infinity mismatch")
    fin = np.isfinite(ref)
    if fin.any():
        err = np.abs(got[fin] - ref[fin])
        bound = TOL_ABS + TOL_REL * np.abs(ref[fin])
        worst = int(np.argmax(err / bound))
        assert (err <= bound).all(), (
            f"{what}: {int((err > bound).sum())} elements out of tolerance; worst err "
            f"{err[worst]:.3e} vs bound {bound[worst]:.3e} (ref {ref[fin][worst]:.6g})")
    return float(np.max(np.abs(got[fin] - ref[fin]))) if fin.any() else 0.0
