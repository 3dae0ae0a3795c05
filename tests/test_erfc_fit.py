"""The erfc approximation the GeGLU kernels use (no GPU).

The constants in csrc/glu.cu must be what csrc/fit_erfc.py produces, and the
approximation evaluated step by step in binary32 (numpy) must stay within the
relative-error bounds include/glu.h states, checked against mpmath.
"""
import os
import re
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "packed_varlen_rope_gb300", "csrc")


def kernel_constants():
    text = open(os.path.join(CSRC, "glu.cu")).read()
    body = re.search(r"kErfcFit\[10\]\s*=\s*\{(.*?)\};", text, flags=re.S).group(1)
    return np.array([float(v.strip().rstrip("f")) for v in body.split(",") if v.strip()], dtype=np.float64)


def fitted(degree=9):
    pytest.importorskip("mpmath")
    sys.path.insert(0, CSRC)
    try:
        import fit_erfc
    finally:
        sys.path.remove(CSRC)
    return fit_erfc.fit(degree)[::-1]


def test_kernel_constants_come_from_the_fit():
    got = kernel_constants()
    want = fitted()
    assert got.shape == want.shape == (10,)
    assert np.allclose(got, want, rtol=1e-8, atol=0)


def _erfc32(z):
    c = kernel_constants().astype(np.float32)
    z = np.asarray(z, dtype=np.float32)
    t = np.float32(1) / (np.float32(1) + np.float32(0.5) * z)
    p = np.full_like(t, c[0])
    for ci in c[1:]:
        p = p * t + ci
    e = (p - z * z) * np.float32(1.4426950408889634)
    return t * np.exp2(e.astype(np.float32)).astype(np.float32)


@pytest.mark.parametrize("xmax,bound", [(6.4, 4e-6), (12.5, 2e-5)])
def test_erfc_approximation_error(xmax, bound):
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    z = np.linspace(0.0, xmax / np.sqrt(2.0), 4001)
    exact = np.array([float(mpmath.erfc(mpmath.mpf(float(v)))) for v in z.astype(np.float32)])
    rel = np.abs(_erfc32(z).astype(np.float64) - exact) / exact
    assert rel.max() < bound, rel.max()
