"""The binary32 constants of the rotation kernels' cos/sin evaluation
(packed_varlen_rope_gb300/csrc/cos_sin.cuh), checked against mpmath at 300 bits:
pi/2 split into three binary32 parts, each the nearest binary32 number to what the
previous parts leave, and 2/pi rounded to nearest.  The series coefficients are 1/n!
written as binary64 quotients in the source and need no table."""
from __future__ import annotations

import os
import re
import struct

import pytest

mpmath = pytest.importorskip("mpmath")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCE = os.path.join(ROOT, "packed_varlen_rope_gb300", "csrc", "cos_sin.cuh")


def _const(name):
    m = re.search(r"constexpr float %s = (-?0x[0-9a-f.]+p[-+]?\d+)f;" % name, open(SOURCE).read())
    assert m, name
    return float.fromhex(m.group(1))


def _rn32(x):
    """Nearest binary32 to the mpmath value x (ties to even), exactly."""
    x = mpmath.mpf(x)
    if x == 0:
        return 0.0
    a = abs(x)
    e = int(mpmath.floor(mpmath.log(a, 2)))
    while mpmath.mpf(2) ** e > a:
        e -= 1
    while mpmath.mpf(2) ** (e + 1) <= a:
        e += 1
    ulp = mpmath.mpf(2) ** (e - 23)
    q = a / ulp
    n = int(mpmath.floor(q))
    rem = q - n
    if rem > 0.5 or (rem == 0.5 and n % 2 == 1):
        n += 1
    return float(mpmath.sign(x) * n * ulp)


def _is_binary32(v):
    return struct.unpack("<f", struct.pack("<f", v))[0] == v


def test_pi_over_2_split():
    mpmath.mp.prec = 300
    pio2 = mpmath.pi / 2
    p1, p2, p3 = _const("kPio2_1"), _const("kPio2_2"), _const("kPio2_3")
    assert all(_is_binary32(v) for v in (p1, p2, p3))
    assert p1 == _rn32(pio2)
    assert p2 == _rn32(pio2 - p1)
    assert p3 == _rn32(pio2 - p1 - p2)
    residual = abs(pio2 - p1 - p2 - p3)
    assert residual < mpmath.mpf(2) ** -76          # 72 bits of pi/2 and a little more
    mpmath.mp.prec = 53


def test_two_over_pi_and_limits():
    mpmath.mp.prec = 300
    c1 = _const("kTwoOverPi_1")
    assert c1 == _rn32(2 / mpmath.pi)
    assert _const("kTwoOverPi_2") == _rn32(2 / mpmath.pi - c1)
    mpmath.mp.prec = 53
    assert _const("kFastLimit") == 2.0 ** 24
    assert _const("kTinyAngle") == 2.0 ** -13
    # below 2^-13, cos rounds to 1 and sin to the angle itself: 1 - x^2/2 stays above the
    # midpoint 1 - 2^-25 under 1, and x - x^3/6 within a quarter unit of x
    x = 2.0 ** -13
    assert x * x / 2 < 2.0 ** -26 and x * x / 6 < 2.0 ** -26


def test_worst_case_reduction_distance(tmp_path):
    """The closest a binary32 angle in [pi/4, 2^24) comes to a multiple of pi/2 (the
    smallest magnitude of the reduced argument): every k = 1 .. 2^24 * 2/pi is walked
    with k * pi/2 in 100-bit fixed point (a small C program, 128-bit integers) and the
    distance to the nearest binary32 number taken.  About 2^-27.8, at k = 161: the
    reduction's absolute error (below 2^-45) stays 2^-17 below every reduced argument."""
    import subprocess

    mpmath.mp.prec = 300
    P = int(mpmath.floor(mpmath.pi / 2 * mpmath.mpf(2) ** 100))
    mpmath.mp.prec = 53
    src = tmp_path / "worst.c"
    src.write_text(r"""
#include <math.h>
#include <stdio.h>
typedef unsigned __int128 u128;
int main(void) {
    const u128 P = ((u128)%dull << 64) | (u128)%dull;
    u128 best = ~(u128)0; long best_k = 0;
    const long kmax = (long)(16777216.0 * 2.0 / M_PI) + 2;
    for (long k = 1; k <= kmax; ++k) {
        const u128 x = (u128)k * P;
        const int sh = ilogb((double)k * M_PI_2) - 23 + 100;
        const u128 ulp = (u128)1 << sh, rem = x & (ulp - 1);
        const u128 d = rem < ulp - rem ? rem : ulp - rem;
        if (d < best) { best = d; best_k = k; }
    }
    printf("%%ld %%.17g\n", best_k, ldexp((double)best, -100));
    return 0;
}
""" % (P >> 64, P & ((1 << 64) - 1)))
    exe = tmp_path / "worst"
    subprocess.check_call(["gcc", "-O2", str(src), "-o", str(exe), "-lm"])
    k, dist = subprocess.check_output([str(exe)], text=True).split()
    assert int(k) == 161
    assert 2.0 ** -28 < float(dist) < 2.0 ** -27.5
