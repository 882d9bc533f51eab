"""Host-side checks of constant tables compiled into the CUDA kernels (no GPU needed).

The TMA scan kernel computes softplus(v) = max(v, 0) + log1p(e), e = exp(-|v|) in (0, 1], with
log1p(e) = e * q(e) and q a degree-7 polynomial whose coefficients are written in
csrc/scan_fast.cuh (kLog1pPoly). These tests read the table from the source and hold it to the
accuracy the kernel's comment states, evaluated the way the kernel evaluates it (Horner's rule in
fp32), against numpy's float64 log1p and logaddexp.
"""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(__file__), "..", "selective_state_space_127_b300", "csrc", "scan_fast.cuh")


def _log1p_poly():
    text = open(SRC).read()
    m = re.search(r"kLog1pPoly\[8\]\s*=\s*\{([^}]*)\}", text)
    assert m, "kLog1pPoly table not found"
    vals = [float(v.strip().rstrip("f")) for v in m.group(1).split(",") if v.strip()]
    assert len(vals) == 8
    return np.array(vals, dtype=np.float32)


def _horner_f32(coef, e):
    e = e.astype(np.float32)
    q = np.full_like(e, coef[0])
    for c in coef[1:]:
        q = (q * e + c).astype(np.float32)
    return (q * e).astype(np.float32)


def test_log1p_polynomial_relative_error_below_4e7_on_the_unit_interval():
    coef = _log1p_poly()
    e = np.concatenate([np.linspace(0.0, 1.0, 400001)[1:], np.logspace(-30, -1, 20001)])
    approx = _horner_f32(coef, e).astype(np.float64)
    exact = np.log1p(e.astype(np.float32).astype(np.float64))
    rel = np.abs(approx - exact) / exact
    assert rel.max() < 4e-7, rel.max()


def test_log1p_polynomial_keeps_relative_accuracy_as_e_goes_to_zero():
    """log1p(e) ~ e for tiny e: the polynomial's constant term is 1 to within 2e-7, so e q(e)
    never loses the relative accuracy a direct log(1 + e) would lose to cancellation."""
    coef = _log1p_poly()
    e = np.array([1e-38, 1e-20, 1e-10, 2.0 ** -24, 2.0 ** -12], dtype=np.float32)
    approx = _horner_f32(coef, e).astype(np.float64)
    rel = np.abs(approx - np.log1p(e.astype(np.float64))) / np.log1p(e.astype(np.float64))
    assert rel.max() < 4e-7


def test_softplus_from_the_polynomial_matches_logaddexp():
    """softplus(v) = max(v, 0) + e q(e), e = exp(-|v|), over the range of delta + bias the
    workloads produce and beyond, with e taken exactly (the kernel's SFU exp adds its own
    ~2^-22 relative error on top)."""
    coef = _log1p_poly()
    v = np.linspace(-40.0, 40.0, 200001)
    e = np.exp(-np.abs(v))
    sp = np.maximum(v, 0.0) + _horner_f32(coef, e).astype(np.float64)
    ref = np.logaddexp(0.0, v)
    rel = np.abs(sp - ref) / ref
    assert rel.max() < 5e-7, rel.max()


def test_a_perturbed_coefficient_fails_the_bound():
    """The bound bites: a one-part-in-10^4 change to the e^6 coefficient breaks it."""
    coef = _log1p_poly().copy()
    coef[1] *= np.float32(1.0001)
    e = np.linspace(0.0, 1.0, 100001)[1:]
    approx = _horner_f32(coef, e).astype(np.float64)
    rel = np.abs(approx - np.log1p(e)) / np.log1p(e)
    assert rel.max() > 4e-7
