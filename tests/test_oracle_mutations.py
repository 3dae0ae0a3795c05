"""Plant plausible slips in a copy of the oracle and check that a pin catches each one.

Every mutant is built from a textual edit of ``oracle/rope_oracle.c`` in a temporary
directory, on the CPU; the committed oracle is never modified.
"""
import os
import shutil

import pytest

import oracle
import oracle_pins

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
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutant_is_caught(tmp_path, name):
    pytest.importorskip("mpmath")
    old, new = MUTATIONS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, "mutation anchor not found: " + old
    mutant_src = tmp_path / "rope_oracle_mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(mutant_src), str(tmp_path / ("librope_oracle_%s.so" % name.replace("-", "_"))))
    mutant = oracle.Oracle(lib)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, "no pin caught mutation " + name
