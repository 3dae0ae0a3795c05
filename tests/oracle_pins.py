"""Checks that pin the CPU oracle to facts fixed outside itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises ``AssertionError`` when
the oracle breaks a fact that the source pages or plain mathematics fix.  They are
collected by ``test_oracle_pins.py`` and re-run against deliberately broken builds of
the oracle by ``test_oracle_mutations.py``, which shows that a plausible slip anywhere
in the oracle trips at least one of them.

What pins what:

* block matrix R of the unsloth.ai page ("Kernel Triton QK RoPE fusionné avec
  packing", backward note; ``tests/golden/rotation_blocks.txt``) -> sign, pairing and
  rounding of the rotation, forward and backward (``pin_matrix``);
* closed forms of the inverse frequencies (powers of ten and of two) -> R3;
* cos/sin evaluated by mpmath at 256 bits, rounded to binary32 by exact comparison
  -> R4/R5 (``pin_cos_sin_mpmath``);
* position 0 is the identity; pair norms are kept; bwd(fwd(x)) == x up to rounding;
  <R(m)q, R(n)k> depends on m - n only -> invariants of any rotation embedding;
* numpy ``searchsorted`` positions, packed == each sample alone, padded == packed
  -> the position reset of the "Packing non contaminé" section;
* torch's CPU bf16 conversion -> round to nearest even;
* mpmath (256 bits) values and derivatives, torch's float64 silu/gelu, and a gradient
  check of the backward -> the SwiGLU/GeGLU oracle (``pin_glu_*``);
* the TRL page's worked rescale (factor 4: position 100,000 reads as 25,000, and the
  163,840 wanted positions map onto the 40,960 trained ones) -> the linear position
  scale (``pin_position_scale``).
"""
from __future__ import annotations

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- helpers

def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return bits_to_f32(bits).astype(np.float64)


def random_bf16_bits(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    """bf16 bit patterns of N(0, scale^2) draws, rounded to nearest even (via torch)."""
    import torch

    f = torch.from_numpy((rng.standard_normal(size=shape) * scale).astype(np.float32))
    return f.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def ulp_bf16(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (normal range; the subnormal spacing below it)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 7)


def load_rotation_blocks():
    """Parse the printed block matrices R and R^T into {name: 2x2 list of block codes}."""
    blocks = {}
    with open(os.path.join(GOLDEN, "rotation_blocks.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, row, b0, b1 = line.split()
            blocks.setdefault(name, [None, None])[int(row)] = [b0, b1]
    return blocks


def block_matrix(code, d: int) -> np.ndarray:
    h = d // 2
    eye = np.eye(h)
    val = {"0": np.zeros((h, h)), "I": eye, "-I": -eye}
    return np.block([[val[code[0][0]], val[code[0][1]]], [val[code[1][0]], val[code[1][1]]]])


def nearest_f32(v) -> np.float32:
    """Round an mpmath number to the nearest binary32, ties to even, by exact comparison."""
    import mpmath

    f = np.float32(float(v))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    best, best_err = None, None
    for c in cands:
        err = abs(mpmath.mpf(float(c)) - v)
        if best is None or err < best_err:
            best, best_err = c, err
        elif err == best_err and (int(np.float32(c).view(np.uint32)) & 1) == 0:
            best = c
    return np.float32(best)


# ---------------------------------------------------------------- pins

def pin_positions(o) -> None:
    # Hand example: the tiny workload's pack, lengths {5, 17, 33, 9}.
    cu = np.array([0, 5, 22, 55, 64], dtype=np.int32)
    exp = np.concatenate([np.arange(n) for n in (5, 17, 33, 9)]).astype(np.int32)
    assert np.array_equal(o.positions(cu, 64), exp)
    # Empty sample and tokens past the last boundary.
    assert o.positions([0, 3, 3, 5], 7).tolist() == [0, 1, 2, 0, 1, -1, -1]
    # Random packs, against numpy's binary search over the sample starts.
    rng = np.random.Generator(np.random.PCG64(11))
    for _ in range(200):
        n = int(rng.integers(1, 12))
        lengths = rng.integers(0, 9, size=n)
        lengths[rng.random(n) < 0.25] = 0
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
        T = int(cu[-1] + rng.integers(0, 4))
        t = np.arange(T)
        s = np.searchsorted(cu[:-1], t, side="right") - 1
        exp = np.where(t < cu[-1], t - cu[s], -1)
        assert np.array_equal(o.positions(cu, T), exp.astype(np.int32))


def pin_inv_freq(o) -> None:
    # theta^(-2j/d) with exact decimal or binary results.
    cases = [
        (1.0e4, 8, [1.0, 0.1, 0.01, 0.001]),
        (1.0e6, 12, [1.0, 0.1, 0.01, 1e-3, 1e-4, 1e-5]),
        (65536.0, 32, [2.0 ** -j for j in range(16)]),
        (5.0e5, 4, [1.0, 5.0e5 ** -0.5]),
    ]
    for theta, d, exp in cases:
        got = o.inv_freq(theta, d)
        want = np.array([np.float32(repr(v)) for v in exp], dtype=np.float32)
        assert np.array_equal(got, want), (theta, d, got, want)
    # 1e4^(-1/2) and 1e6^(-1/2) sit at j = d/4 of the head dims the workloads use.
    assert o.inv_freq(1.0e4, 64)[16] == np.float32("0.01")
    assert o.inv_freq(1.0e6, 128)[32] == np.float32("0.001")
    assert np.all(np.diff(o.inv_freq(1.0e6, 128)) < 0)


def pin_cos_sin_mpmath(o) -> None:
    import mpmath

    mpmath.mp.prec = 256
    exact = mismatch = 0
    for theta, d in ((1.0e4, 64), (1.0e6, 128), (5.0e5, 128)):
        w = o.inv_freq(theta, d)
        for pos in (0, 1, 2, 7, 100, 4095, 65535, 524287, 1048575):
            c, s = o.cos_sin(pos, theta, d)
            for j in range(0, d // 2, 3):
                phi = nearest_f32(mpmath.mpf(pos) * mpmath.mpf(float(w[j])))
                ce = nearest_f32(mpmath.cos(mpmath.mpf(float(phi))))
                se = nearest_f32(mpmath.sin(mpmath.mpf(float(phi))))
                for got, want in ((c[j], ce), (s[j], se)):
                    if got == want:
                        exact += 1
                    else:
                        mismatch += 1
                        # Only a value within ~2^-50 of a rounding boundary may differ.
                        assert abs(int(np.float32(got).view(np.int32)) -
                                   int(np.float32(want).view(np.int32))) <= 1, (pos, j, got, want)
    assert mismatch <= 1, mismatch
    assert o.cos_sin(0, 1.0e6, 128)[0].tolist() == [1.0] * 64


def pin_identity_pos0(o) -> None:
    rng = np.random.Generator(np.random.PCG64(12))
    x = random_bf16_bits(rng, (5, 3, 64))
    pos = np.zeros(5, dtype=np.int32)
    assert np.array_equal(o.rope_rows(x, pos, 1.0e4), x)
    assert np.array_equal(o.rope_rows(x, pos, 1.0e4, bwd=True), x)


def pin_matrix(o) -> None:
    blocks = load_rotation_blocks()
    rng = np.random.Generator(np.random.PCG64(13))
    for d in (4, 8, 64):
        h = d // 2
        R = block_matrix(blocks["R"], d)
        RT = block_matrix(blocks["RT"], d)
        assert np.array_equal(RT, R.T)
        for theta in (1.0e4, 1.0e6):
            rows = 40
            x = random_bf16_bits(rng, (rows, 2, d))
            pos = rng.integers(0, 65, size=rows).astype(np.int32)
            for bwd, M in ((False, R), (True, RT)):
                y = bits_to_f64(o.rope_rows(x, pos, theta, bwd=bwd))
                for r in range(rows):
                    c, s = o.cos_sin(int(pos[r]), theta, d)
                    cf = np.concatenate([c, c]).astype(np.float64)
                    sf = np.concatenate([s, s]).astype(np.float64)
                    xr = bits_to_f64(x[r])                       # [2, d]
                    want = xr * cf + (xr @ M) * sf
                    mag = np.abs(xr) + np.abs(np.roll(xr, h, axis=1))
                    bound = 0.5 * ulp_bf16(np.maximum(np.abs(want), np.abs(y[r]))) + 2.0 ** -22 * mag
                    err = np.abs(y[r] - want)
                    assert np.all(err <= bound), (d, theta, bwd, r, float(np.max(err - bound)))


def pin_pair_norm(o) -> None:
    rng = np.random.Generator(np.random.PCG64(14))
    x = random_bf16_bits(rng, (64, 4, 128))
    pos = rng.integers(0, 1 << 20, size=64).astype(np.int32)
    y = bits_to_f64(o.rope_rows(x, pos, 1.0e6))
    xf = bits_to_f64(x)
    nx = np.hypot(xf[..., :64], xf[..., 64:])
    ny = np.hypot(y[..., :64], y[..., 64:])
    assert np.all(np.abs(ny - nx) <= 2.0 ** -7 * nx + 1e-30)


def pin_roundtrip(o) -> None:
    rng = np.random.Generator(np.random.PCG64(15))
    x = random_bf16_bits(rng, (64, 4, 128))
    pos = rng.integers(0, 1 << 20, size=64).astype(np.int32)
    back = bits_to_f64(o.rope_rows(o.rope_rows(x, pos, 1.0e6), pos, 1.0e6, bwd=True))
    xf = bits_to_f64(x)
    mag = np.abs(xf) + np.abs(np.roll(xf, 64, axis=-1))
    assert np.all(np.abs(back - xf) <= 2.0 ** -7 * mag)
    # and the forward alone is not the identity away from position 0
    assert not np.array_equal(o.rope_rows(x, pos, 1.0e6), x)


def pin_packed_equals_alone(o) -> None:
    rng = np.random.Generator(np.random.PCG64(16))
    lengths = [7, 0, 31, 1, 64, 0, 9]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1]) + 3
    x = random_bf16_bits(rng, (T, 3, 16))
    for bwd in (False, True):
        packed = o.rope_packed(x, cu, 1.0e4, bwd=bwd)
        for s, L in enumerate(lengths):
            a, b = int(cu[s]), int(cu[s + 1])
            alone = o.rope_packed(x[a:b], np.array([0, L], dtype=np.int32), 1.0e4, bwd=bwd)
            assert np.array_equal(packed[a:b], alone)
        assert np.array_equal(packed[cu[-1]:], x[cu[-1]:])        # outside: untouched


def pin_padded_equals_packed(o) -> None:
    rng = np.random.Generator(np.random.PCG64(17))
    lengths = [int(v) for v in rng.integers(4, 32, size=5)]
    pad_to = 32
    x_pad = random_bf16_bits(rng, (5 * pad_to, 2, 32))
    cu_pad = np.arange(6, dtype=np.int32) * pad_to
    valid = np.concatenate([np.arange(b * pad_to, b * pad_to + L) for b, L in enumerate(lengths)])
    cu_pack = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    y_pad = o.rope_packed(x_pad, cu_pad, 5.0e5)
    y_pack = o.rope_packed(x_pad[valid], cu_pack, 5.0e5)
    assert np.array_equal(y_pad[valid], y_pack)


def pin_relative_position(o) -> None:
    rng = np.random.Generator(np.random.PCG64(18))
    d, theta = 64, 1.0e4
    moved = 0
    for _ in range(60):
        q = random_bf16_bits(rng, (1, 1, d))
        k = random_bf16_bits(rng, (1, 1, d))
        m, n, shift = (int(v) for v in rng.integers(0, 2000, size=3))

        def dot(pm, pn):
            qr = bits_to_f64(o.rope_rows(q, np.array([pm], np.int32), theta))[0, 0]
            kr = bits_to_f64(o.rope_rows(k, np.array([pn], np.int32), theta))[0, 0]
            return float(qr @ kr)

        scale = float(np.linalg.norm(bits_to_f64(q)) * np.linalg.norm(bits_to_f64(k)))
        base = dot(m, n)
        assert abs(base - dot(m + shift, n + shift)) <= 2.0 ** -6 * scale
        if abs(base - dot(m, n + 37)) > 2.0 ** -4 * scale:
            moved += 1
    assert moved >= 30          # the product does depend on m - n


def pin_bf16_rounding(o) -> None:
    import torch

    special = [0.0, -0.0, 1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8),
               1.0 + 2.0 ** -8 + 2.0 ** -20, 2.0 ** -130, -(2.0 ** -133) * 3, 3.0e38, -3.0e38,
               float("inf"), float("-inf"), 65504.0, 1.0e-40]
    rng = np.random.Generator(np.random.PCG64(19))
    vals = np.concatenate([np.array(special, dtype=np.float32),
                           (rng.standard_normal(20000) * np.exp2(rng.integers(-20, 20, 20000)))
                           .astype(np.float32)])
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([o.float_to_bf16_bits(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, want)


def pin_position_scale(o) -> None:
    import mpmath

    rng = np.random.Generator(np.random.PCG64(20))
    x = random_bf16_bits(rng, (4, 3, 128))
    # the page's worked example (tests/golden/position_rescale.txt: TRL "training
    # beyond 1M tokens", YaRN section); a power-of-two factor gives identical bits
    rows = [tuple(int(v) for v in line.split()) for line in
            open(os.path.join(GOLDEN, "position_rescale.txt")) if line.strip() and not line.startswith("#")]
    assert rows and all(f == 163840 // 40960 for f, _, _ in rows)
    for factor, pos, rescaled in rows:
        assert pos == rescaled * factor
    positions = np.array([p for _, p, _ in rows] + [4, 0], np.int32)
    expected = np.array([r for _, _, r in rows] + [1, 0], np.int32)
    for theta in (1.0e6, 1.0e4):
        for bwd in (False, True):
            scaled = o.rope_rows(x, positions, theta, bwd=bwd, scale=float(rows[0][0]))
            plain = o.rope_rows(x, expected, theta, bwd=bwd)
            assert np.array_equal(scaled, plain)
    # frequencies divided by the scale: exact for powers of two ...
    for d in (8, 64, 128):
        assert np.array_equal(o.inv_freq(1.0e6, d, 4.0), o.inv_freq(1.0e6, d) / np.float32(4.0))
        assert np.array_equal(o.inv_freq(1.0e6, d, 1.0), o.inv_freq(1.0e6, d))
    # ... and rounded once otherwise (mpmath, within one binary32 step)
    mpmath.mp.prec = 256
    w = o.inv_freq(5.0e5, 64, 2.5)
    for j in range(32):
        exact = mpmath.power(mpmath.mpf(5.0e5), mpmath.mpf(-2 * j) / 64) / mpmath.mpf(2.5)
        want = nearest_f32(exact)
        assert abs(int(np.float32(w[j]).view(np.int32)) - int(want.view(np.int32))) <= 1, (j, w[j], want)
    # a scaled position is not the plain one
    assert not np.array_equal(o.rope_rows(x, np.array([100000] * 4, np.int32), 1.0e6, scale=4.0),
                              o.rope_rows(x, np.array([100000] * 4, np.int32), 1.0e6))


# ---------------------------------------------------------------- gated MLP activations

GLU_KINDS = ("swiglu", "geglu", "geglu_tanh")


def _mp_act(kind, x):
    import mpmath

    # high-precision values; erfc and 1/(1 + exp(-2u)) keep the far tails exact, where
    # 1 + erf and 1 + tanh would cancel even at 256 bits
    x = mpmath.mpf(x)
    if kind == "swiglu":
        return x / (1 + mpmath.exp(-x))
    if kind == "geglu":
        return x * mpmath.erfc(-x / mpmath.sqrt(2)) / 2
    u = mpmath.sqrt(2 / mpmath.pi) * (x + mpmath.mpf("0.044715") * x ** 3)
    return x / (1 + mpmath.exp(-2 * u))


def _mp_dact_terms(kind, x):
    """Sum of the absolute values of the terms of act'(x) (a scale for its rounding)."""
    import mpmath

    x = mpmath.mpf(x)
    sig = lambda t: 1 / (1 + mpmath.exp(-t))  # noqa: E731
    if kind == "swiglu":
        return float(sig(x) * (1 + abs(x) * sig(-x)))
    if kind == "geglu":
        return float(mpmath.erfc(-x / mpmath.sqrt(2)) / 2 + abs(x) * mpmath.exp(-x * x / 2) / mpmath.sqrt(2 * mpmath.pi))
    u = mpmath.sqrt(2 / mpmath.pi) * (x + mpmath.mpf("0.044715") * x ** 3)
    return float(sig(2 * u) + 2 * abs(x) * sig(2 * u) * sig(-2 * u) * mpmath.sqrt(2 / mpmath.pi)
                 * (1 + 3 * mpmath.mpf("0.044715") * x * x))


def nearest_bf16_bits(v) -> int:
    """Nearest bf16 (ties to even) of an mpmath/float value, by exact comparison of
    neighbouring bf16 values."""
    import mpmath

    f = np.float32(float(v))
    b = int(f.view(np.uint32)) >> 16
    best, best_err = None, None
    for c in (b - 1, b, b + 1, b + 2):
        c &= 0xFFFF
        cv = bits_to_f64(np.array([c], np.uint16))[0]
        if not np.isfinite(cv):
            continue
        err = abs(mpmath.mpf(cv) - mpmath.mpf(v))
        if best is None or err < best_err or (err == best_err and c % 2 == 0):
            best, best_err = c, err
    return best


def pin_glu_activation(o) -> None:
    """act and act' against mpmath at 256 bits, mpmath numerical derivatives, and torch's
    float64 silu / gelu / gelu(tanh) as independent library routines."""
    import mpmath
    import torch

    mpmath.mp.prec = 256
    xs = [0.0, 1.0, -1.0, 0.5, -2.75, 3.25, 8.0, -8.0, 20.0, -20.0, -12.5, -30.0, 1e-3, -1e-3,
          0.044715, -1.2784645, -6.0, 6.0, -89.0, -720.0]
    for kind in GLU_KINDS:
        assert o.glu_activation(kind, 0.0) == (0.0, 0.5)
        for x in xs:
            a, da = o.glu_activation(kind, x)
            ea = _mp_act(kind, x)
            eda = mpmath.diff(lambda t: _mp_act(kind, t), mpmath.mpf(x))
            # relative accuracy everywhere (the tails included), not just an absolute one
            # relative down to the smallest normal binary64 (2^-1022); below it the
            # subnormals carry fewer bits, so the bound there is absolute
            assert abs(a - ea) <= 1e-13 * max(abs(ea), 2.0 ** -1022), (kind, x, a, ea)
            # act' is a sum of terms; where it crosses zero only the terms' size bounds it
            assert abs(da - eda) <= 1e-12 * max(abs(eda), 2.0 ** -1022) + 1e-15 * _mp_dact_terms(kind, x), \
                (kind, x, da, eda)
        # torch's float64 formulas cancel in the far tails, so compare them where they hold
        core = [x for x in xs if abs(x) <= 4.0]
        t = torch.tensor(core, dtype=torch.float64)
        ref = {"swiglu": torch.nn.functional.silu(t), "geglu": torch.nn.functional.gelu(t),
               "geglu_tanh": torch.nn.functional.gelu(t, approximate="tanh")}[kind]
        got = np.array([o.glu_activation(kind, x)[0] for x in core])
        assert np.allclose(got, ref.numpy(), rtol=1e-12, atol=1e-300)
    # SiLU at ln 3: sigmoid is exactly 3/4
    a, _ = o.glu_activation("swiglu", float(np.log(3.0)))
    assert abs(a - 0.75 * np.log(3.0)) <= 4 * np.spacing(a)


def pin_double_to_bf16(o) -> None:
    import mpmath

    rng = np.random.Generator(np.random.PCG64(21))
    vals = list(rng.standard_normal(3000) * np.exp2(rng.integers(-140, 120, 3000)))
    vals += [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 1.0 + 2.0 ** -8 + 2.0 ** -40,
             2.0 ** -134, 3 * 2.0 ** -135, 2.0 ** -126 * (1 - 2.0 ** -9), 0.0, -0.0,
             float(np.float32(1.0 + 2.0 ** -8)) + 2.0 ** -30]
    for v in vals:
        got = o.double_to_bf16_bits(v)
        if v == 0.0:
            assert got == (0x8000 if np.signbit(v) else 0)
            continue
        assert got == nearest_bf16_bits(mpmath.mpf(v)), (v, hex(got))


def pin_glu_gradient(o) -> None:
    """The backward is the gradient of L = sum(dh * act(e) * g): de and dg against
    mpmath derivatives of L, rounded once to bf16."""
    import mpmath

    mpmath.mp.prec = 128
    rng = np.random.Generator(np.random.PCG64(22))
    n = 48
    e, g, dh = (random_bf16_bits(rng, (n,), 2.0) for _ in range(3))
    ef, gf, dhf = bits_to_f64(e), bits_to_f64(g), bits_to_f64(dh)
    for kind in GLU_KINDS:
        de, dg = o.glu_bwd(kind, dh, e, g)
        h = o.glu_fwd(kind, e, g)
        for i in range(n):
            L = lambda ee, gg: mpmath.mpf(dhf[i]) * _mp_act(kind, ee) * gg  # noqa: E731
            want_de = mpmath.diff(lambda t: L(t, mpmath.mpf(gf[i])), mpmath.mpf(ef[i]))
            want_dg = mpmath.diff(lambda t: L(mpmath.mpf(ef[i]), t), mpmath.mpf(gf[i]))
            assert int(de[i]) == nearest_bf16_bits(want_de), (kind, i)
            assert int(dg[i]) == nearest_bf16_bits(want_dg), (kind, i)
            assert int(h[i]) == nearest_bf16_bits(_mp_act(kind, ef[i]) * mpmath.mpf(gf[i])), (kind, i)


ALL_PINS = [pin_positions, pin_inv_freq, pin_cos_sin_mpmath, pin_identity_pos0, pin_matrix,
            pin_pair_norm, pin_roundtrip, pin_packed_equals_alone, pin_padded_equals_packed,
            pin_relative_position, pin_bf16_rounding, pin_position_scale,
            pin_glu_activation, pin_double_to_bf16, pin_glu_gradient]
