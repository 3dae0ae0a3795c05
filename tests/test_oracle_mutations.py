"""Plant plausible slips in a copy of the oracle and check that a pin catches each one.

Every mutant is built from a textual edit of ``oracle/rope_oracle.c`` in a temporary
directory, on the CPU; the committed oracle is never modified.
"""
import os

import pytest

import oracle
import oracle_pins

GLU = "glu_oracle.c"

MUTATIONS = {
    "lo-sign": ("float lo = ac - bs;", "float lo = ac + bs;"),
    "hi-sign": ("float hi = bc + as;", "float hi = bc - as;"),
    "halves-swapped": ("yh[i + h] = oracle_float_to_bf16(hi);", "yh[i + h] = oracle_float_to_bf16(lo);"),
    "pair-neighbour": ("float b = bf16_bits_to_float(xh[i + h]);",
                       "float b = bf16_bits_to_float(xh[i ^ 1]);"),
    "freq-exponent": ("double e = -(2.0 * (double)j) / (double)d;",
                      "double e = -((double)j) / (double)d;"),
    "freq-sign": ("double e = -(2.0 * (double)j) / (double)d;",
                  "double e = (2.0 * (double)j) / (double)d;"),
    "angle-fp64": ("float phi = (float)pos * w[j];", "double phi = (double)pos * (double)w[j];"),
    "cos-sin-swapped": ("c_out[j] = (float)cos((double)phi);", "c_out[j] = (float)sin((double)phi);"),
    "bf16-truncate": ("u += 0x7fffu + keep_lsb;", "u += 0u;"),
    "bf16-ties-away": ("u += 0x7fffu + keep_lsb;", "u += 0x8000u;"),
    "no-position-reset": ("pos_out[t] = (int32_t)(t - start);", "pos_out[t] = (int32_t)t;"),
    "position-off-by-one": ("pos_out[t] = (int32_t)(t - start);", "pos_out[t] = (int32_t)(t - start + 1);"),
    "bwd-sign-ignored": ("float sn = bwd ? -s[i] : s[i];", "float sn = s[i];"),
    "theta-ignored": ("w_out[j] = (float)(pow(theta, e) / scale);", "w_out[j] = (float)(pow(10000.0, e) / scale);"),
    "scale-multiplies": ("w_out[j] = (float)(pow(theta, e) / scale);", "w_out[j] = (float)(pow(theta, e) * scale);"),
    "scale-ignored": ("w_out[j] = (float)(pow(theta, e) / scale);", "w_out[j] = (float)pow(theta, e);"),
    # SwiGLU / GeGLU oracle
    "glu-sigmoid-sign": ("return x >= 0.0 ? 1.0 / (1.0 + t) : t / (1.0 + t);", "return x >= 0.0 ? t / (1.0 + t) : 1.0 / (1.0 + t);", GLU),
    "glu-silu-derivative": ("*dact = s * (1.0 + x * sigmoid(-x));", "*dact = s * (1.0 + x * sigmoid(x));", GLU),
    "glu-erf-argument": ("0.5 * erfc(-x * kInvSqrt2);", "0.5 * erfc(-x * kSqrt2OverPi);", GLU),
    "glu-erfc-sign": ("0.5 * erfc(-x * kInvSqrt2);", "0.5 * erfc(x * kInvSqrt2);", GLU),
    "glu-tanh-form-factor": ("double sp = sigmoid(2.0 * u), sm = sigmoid(-2.0 * u);", "double sp = sigmoid(u), sm = sigmoid(-u);", GLU),
    "glu-gelu-derivative-term": ("*dact = Phi + x * phi;", "*dact = Phi;", GLU),
    "glu-tanh-cubic": ("(x + kGeluTanhC * x * x * x)", "(x + kGeluTanhC * x * x)", GLU),
    "glu-dg-uses-derivative": ("dg[i] = double_to_bf16(dhi * a);", "dg[i] = double_to_bf16(dhi * da);", GLU),
    "glu-de-drops-g": ("de[i] = double_to_bf16(dhi * gi * da);", "de[i] = double_to_bf16(dhi * da);", GLU),
    "glu-round-truncates": ("double r = ldexp(nearbyint(ldexp(v, -q)), q);", "double r = ldexp(trunc(ldexp(v, -q)), q);", GLU),
    "glu-fwd-uses-derivative": ("h[i] = double_to_bf16(a * bf16_to_double(g[i]));", "h[i] = double_to_bf16(da * bf16_to_double(g[i]));", GLU),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutant_is_caught(tmp_path, name):
    pytest.importorskip("mpmath")
    old, new, *where = MUTATIONS[name]
    target = where[0] if where else "rope_oracle.c"
    sources = []
    for path in oracle.SOURCES:
        text = open(path).read()
        if os.path.basename(path) == target:
            assert text.count(old) == 1, "mutation anchor not found: " + old
            text = text.replace(old, new)
        out = tmp_path / os.path.basename(path)
        out.write_text(text)
        sources.append(str(out))
    lib = oracle.compile_source(sources, str(tmp_path / ("liboracle_%s.so" % name.replace("-", "_"))))
    mutant = oracle.Oracle(lib)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, "no pin caught mutation " + name
