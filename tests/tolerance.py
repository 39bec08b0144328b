"""Parity checks of GPU results against the oracle, with the stated tolerances.

* binary32 outputs: max |gpu - oracle| <= 2e-5 (oracle value in double).
* binary16 / bfloat16 outputs: within 1 ulp of the oracle's value rounded to
  the type (ulp distance of the bit patterns).
  LayerNorm/BatchNorm outputs y = t*gamma + beta, t = (x - mean)*rstd, can be
  tiny because of cancellation between t*gamma and beta; no binary32
  evaluation is within 1 ulp of such a result.  For those elements only, the
  bound is the binary32 evaluation error, 2^-20 * (|t*gamma| + |beta| + |gamma|)
  (16 unit roundoffs of each term): |t*gamma| carries the relative error of
  rstd and of the products, |beta| the final rounding, and |gamma| the error
  of a binary32 mean, which is a few roundoffs of the spread (one standardized
  unit, times gamma).  The test reports how many elements used this bound.
* residual_out: bit-exact.
* statistics (mean, rstd, save_*, running_*): relative 1e-5, and for a mean
  absolute 1e-5 * (|mean| + sqrt(var)).
* BatchNorm backward dx = gamma*rstd*(dy - s1/cnt - xhat*s2/cnt): the binary32
  evaluation error is a few unit roundoffs of each term plus the error of the
  two channel sums, at most (depth of the summation tree, about 25) unit
  roundoffs of sum|dy| and sum|dy*xhat|.  Bound: |err| <= 1e-5 * S with
  S = |gamma|*rstd*(|dy| + (|s1| + sum|dy|)/cnt + |xhat|*(|s2| + sum|dy*xhat|)/cnt),
  about 5 times that estimate; 16-bit dx may instead be within 1 ulp of the
  oracle rounded.  dbeta, dgamma: |err| <= 1e-5 * sum|dy| and 1e-5 * sum|dy*xhat|.
* Softmax y = exp(x - m) / d in binary32: each expf is within 2 ulp (CUDA's
  documented bound), the row sum d carries at most one roundoff per term a
  thread adds (up to N / 512 = 128 terms in the generic plan at N = 65536)
  plus two exponentials and an add per merge level (about 9 levels), and the
  output adds an exponential, a division and a product: at most about 160
  unit roundoffs (1e-5) in all.  Bound: |err| <= 2e-5 * y + 2^-126 (the
  absolute part covers results below the normal range); binary16/bfloat16 y
  within 1 ulp of the oracle rounded; row_max bit-exact (the max of stored
  values is exact); row_sum relative 2e-5.
"""
import numpy as np

import bits as B

TOL_F32 = 2e-5
CANCEL_REL = 2.0 ** -20
STAT_REL = 1e-5
BWD_REL = 1e-5
SOFTMAX_REL = 2e-5


def check_y(dt, got, ref_bits, ref_wide, affine_scale=None, what="y"):
    """Compare output y; returns a dict of measured errors.  affine_scale, when
    given, is |t*gamma| + |beta| per element (LayerNorm-type outputs)."""
    got = np.asarray(got)
    g64 = B.bits_to_f64(dt, got)
    err = np.abs(g64 - ref_wide)
    if dt == 0:
        m = float(np.max(err)) if err.size else 0.0
        assert m <= TOL_F32, f"{what}: max abs err {m} > {TOL_F32}"
        return {"max_abs_err": m}
    ulps = B.ulp_diff(dt, got, ref_bits)
    bad = ulps > 1
    n_floor = 0
    if np.any(bad):
        assert affine_scale is not None, (
            f"{what}: {int(bad.sum())} elements > 1 ulp (max {int(ulps.max())} ulp)")
        bound = CANCEL_REL * affine_scale[bad]
        over = ~(err[bad] <= bound)  # NaN fails
        assert not np.any(over), (
            f"{what}: {int(over.sum())} elements > 1 ulp and beyond the cancellation bound; "
            f"worst err {float(np.max(err[bad][over]))}")
        n_floor = int(bad.sum())
    return {"max_ulp": int(ulps.max()) if ulps.size else 0, "n_cancel_floor": n_floor,
            "max_abs_err": float(np.max(err)) if err.size else 0.0}


def check_scaled(dt, got, ref_bits, ref_wide, scale, rel, what):
    """|got - oracle| <= rel * scale per element; 16-bit outputs pass as well
    when within 1 ulp of the oracle rounded to the type."""
    got = np.asarray(got)
    g64 = B.bits_to_f64(dt, got)
    err = np.abs(g64 - ref_wide)
    over = ~(err <= rel * scale)  # NaN fails
    if dt != 0 and np.any(over):
        over &= B.ulp_diff(dt, got, ref_bits) > 1
    assert not np.any(over), (
        f"{what}: {int(over.sum())} elements beyond the bound; worst ratio "
        f"{float(np.max(err[over] / (rel * scale[over])))}")
    return {"max_abs_err": float(np.max(err)) if err.size else 0.0,
            "max_err_over_scale": float(np.max(err / scale)) if err.size else 0.0}


def check_softmax(dt, got, ref_bits, ref_wide, what="y"):
    got = np.asarray(got)
    g64 = B.bits_to_f64(dt, got)
    err = np.abs(g64 - ref_wide)
    if dt == 0:
        bound = SOFTMAX_REL * np.abs(ref_wide) + 2.0 ** -126
        over = ~(err <= bound)  # NaN fails
        assert not np.any(over), (
            f"{what}: {int(over.sum())} elements beyond 2e-5 relative; worst "
            f"{float(np.max(err[over] / bound[over]))} x the bound")
        return {"max_rel_err": float(np.max(err / np.maximum(np.abs(ref_wide), 2.0 ** -126)))
                if err.size else 0.0}
    assert not np.any(np.isnan(g64) & ~np.isnan(ref_wide)), f"{what}: NaN where the oracle has none"
    ulps = B.ulp_diff(dt, got, ref_bits)
    assert not np.any(ulps > 1), f"{what}: {int((ulps > 1).sum())} elements > 1 ulp"
    return {"max_ulp": int(ulps.max()) if ulps.size else 0}


def check_stat(got, ref, what, scale=None):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    tol = STAT_REL * (np.abs(ref) if scale is None else scale)
    err = np.abs(got - ref)
    assert np.all(err <= tol), f"{what}: max err {float(np.max(err - tol))} over tolerance"
    return float(np.max(err / np.maximum(tol / STAT_REL, 1e-300))) if err.size else 0.0


def ln_affine_scale(dt, x_bits, mean, rstd, gamma_bits=None, beta_bits=None):
    x = B.bits_to_f64(dt, x_bits)
    t = (x - mean[..., None]) * rstd[..., None]
    g = 1.0 if gamma_bits is None else B.bits_to_f64(dt, gamma_bits)
    b = 0.0 if beta_bits is None else B.bits_to_f64(dt, beta_bits)
    return np.abs(t * g) + np.abs(b) + np.abs(g)
