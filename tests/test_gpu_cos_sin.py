"""The rotation's cos/sin without a table (needs a GB300).

The kernels take c = RN32(cos phi), s = RN32(sin phi) of phi = RN32(pos * w_j) from a
binary32 double-float evaluation when its rounding is certain and from binary64
otherwise.  Checked here:

* every binary32 angle in [2^-20, 2^24) -- each phi the rotation can meet for
  positions below 2^24 and frequencies up to 1 -- gives the bits of the binary64
  evaluation (rope_cos_sin_eval, the same device function the kernels call), and the
  binary32 path alone decides all but a few in a million of them;
* angles outside that range (zero, subnormals, tiny, at or past 2^24, negative,
  infinite, NaN) give the binary64 bits too;
* the rotation without a cache over every position of the 2^20-token sequence equals
  the CPU oracle bit for bit.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import struct

import numpy as np
import pytest

import oracle
from parity_util import to_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from packed_varlen_rope_gb300 import build

    build.build()
    oracle.build()
    return torch.device("cuda:0")


MODES = ("as_rotation", "binary64", "binary32_only")


def _eval(lib, phi, mode):
    return lib.rope_cos_sin_eval(phi, MODES[mode])


def _lib():
    import packed_varlen_rope_gb300 as pr

    return pr


def _f32_bits(v):
    return struct.unpack("<i", struct.pack("<f", v))[0]


def test_every_angle_below_2_24_matches_binary64(dev):
    lib = _lib()
    lo, hi = _f32_bits(2.0 ** -20), _f32_bits(2.0 ** 24)
    chunk = 1 << 25
    total = mismatch = deferred = 0
    for start in range(lo, hi, chunk):
        phi = torch.arange(start, min(hi, start + chunk), dtype=torch.int32, device=dev).view(torch.float32)
        c0, s0 = _eval(lib, phi, 0)
        c1, s1 = _eval(lib, phi, 1)
        c2, s2 = _eval(lib, phi, 2)
        as_i = lambda t: t.view(torch.int32)  # noqa: E731
        mismatch += int((as_i(c0) != as_i(c1)).sum()) + int((as_i(s0) != as_i(s1)).sum())
        decided = ~torch.isnan(c2)
        assert torch.equal(decided, ~torch.isnan(s2))
        assert torch.equal(as_i(c2)[decided], as_i(c1)[decided])
        assert torch.equal(as_i(s2)[decided], as_i(s1)[decided])
        deferred += int((~decided).sum())
        total += phi.numel()
    assert total == hi - lo
    assert mismatch == 0
    print("angles %d, left to binary64 %d (%.3g)" % (total, deferred, deferred / total))
    assert deferred / total < 1e-4


def test_angles_outside_the_fast_range(dev):
    lib = _lib()
    rng = np.random.Generator(np.random.PCG64(77))
    small = rng.integers(1, _f32_bits(2.0 ** -20), size=1 << 20, dtype=np.int64).astype(np.int32)
    big = rng.integers(_f32_bits(2.0 ** 24), 0x7F800000, size=1 << 16, dtype=np.int64).astype(np.int32)
    special = np.array([0, _f32_bits(-0.0), 1, 0x7FFFFF, 0x800000, _f32_bits(2.0 ** -13), _f32_bits(2.0 ** 24),
                        0x7F800000, _f32_bits(-1.0), _f32_bits(-3.0e7), 0x7FC00000, 0xFF800000 - (1 << 32)],
                       dtype=np.int64).astype(np.int32)
    phi = torch.from_numpy(np.concatenate([small, big, special])).to(dev).view(torch.float32)
    c0, s0 = _eval(lib, phi, 0)
    c1, s1 = _eval(lib, phi, 1)
    assert torch.equal(c0.view(torch.int32), c1.view(torch.int32))
    assert torch.equal(s0.view(torch.int32), s1.view(torch.int32))


@pytest.mark.parametrize("theta,d,bwd", [(1.0e6, 128, False), (5.0e5, 64, True), (1.0e4, 128, True)])
def test_no_cache_rotation_every_position(dev, theta, d, bwd):
    """One 1,048,576-token sequence (positions 0 .. 2^20 - 1), one Q and one K head,
    rotated without a cos/sin cache: every element equals the oracle's."""
    import packed_varlen_rope_gb300 as pr
    from packed_varlen_rope_gb300 import workloads as wl

    T = 1 << 20
    q = wl.normal_bf16((T, 1, d), 61, device=dev)
    k = wl.normal_bf16((T, 1, d), 62, device=dev)
    qb, kb = to_bits(q), to_bits(k)
    cu = torch.tensor([0, T], dtype=torch.int32, device=dev)
    (pr.rope_qk_bwd if bwd else pr.rope_qk_fwd)(q, k, cu, theta)
    torch.cuda.synchronize()
    pos = np.arange(T, dtype=np.int32)
    n = len(os.sched_getaffinity(0))
    bounds = np.linspace(0, T, n + 1).astype(np.int64)
    ref_q, ref_k = np.empty_like(qb), np.empty_like(kb)

    def part(i):
        a, b = bounds[i], bounds[i + 1]
        ref_q[a:b] = oracle.rope_rows(qb[a:b], pos[a:b], theta, bwd=bwd)
        ref_k[a:b] = oracle.rope_rows(kb[a:b], pos[a:b], theta, bwd=bwd)

    with cf.ThreadPoolExecutor(n) as ex:
        list(ex.map(part, range(n)))
    assert np.array_equal(to_bits(q), ref_q)
    assert np.array_equal(to_bits(k), ref_k)
