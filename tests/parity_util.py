"""Element-by-element comparison of CUDA results with the CPU oracle.

The bar (floating point): |gpu - ref| <= 2 bf16 ULP of the reference value AND
|gpu - ref| <= 1e-2, where the ULP is taken at m = max(|ref|, 2^-16 * (|a| + |b|)) and
a, b are the two inputs of the element's rotation pair.  The floor only matters under
catastrophic cancellation (|ref| far below |a| + |b|); the number of elements it
admits is reported.  Positions and every index are compared bit for bit.  Bit-level
mismatches are counted as well: with the arithmetic fixed step by step on both sides
they are expected to be zero.
"""
from __future__ import annotations

import numpy as np

from oracle_pins import bits_to_f64, ulp_bf16

ABS_TOL = 1e-2
ULP_TOL = 2.0


def to_bits(t) -> np.ndarray:
    import torch

    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bits(bits: np.ndarray, device):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def compare(got_bits: np.ndarray, ref_bits: np.ndarray, x_bits: np.ndarray) -> dict:
    """Compare [rows, H, d] bf16 bit arrays; x_bits are the inputs of the rotation."""
    assert got_bits.shape == ref_bits.shape == x_bits.shape
    half = x_bits.shape[-1] // 2
    g = bits_to_f64(got_bits)
    r = bits_to_f64(ref_bits)
    x = bits_to_f64(x_bits)
    mag = np.abs(x) + np.abs(np.roll(x, half, axis=-1))
    m = np.maximum(np.abs(r), 2.0 ** -16 * mag)
    both_nan = np.isnan(g) & np.isnan(r)
    same_inf = np.isinf(g) & np.isinf(r) & (np.sign(g) == np.sign(r))
    with np.errstate(invalid="ignore"):
        err = np.abs(g - r)
        ok = ((err <= ULP_TOL * ulp_bf16(m)) & (err <= ABS_TOL)) | both_nan | same_inf
        floor_used = ok & ~both_nan & ~same_inf & (err > ULP_TOL * ulp_bf16(r))
    finite_err = np.where(ok & ~both_nan & ~same_inf, err, 0.0)
    return {
        "n": int(got_bits.size),
        "bit_mismatch": int(np.count_nonzero(got_bits != ref_bits)),
        "violations": int(np.count_nonzero(~ok)),
        "floor_admitted": int(np.count_nonzero(floor_used)),
        "max_abs_err": float(finite_err.max()) if finite_err.size else 0.0,
    }


def merge(a: dict, b: dict) -> dict:
    if not a:
        return dict(b)
    return {"n": a["n"] + b["n"], "bit_mismatch": a["bit_mismatch"] + b["bit_mismatch"],
            "violations": a["violations"] + b["violations"],
            "floor_admitted": a["floor_admitted"] + b["floor_admitted"],
            "max_abs_err": max(a["max_abs_err"], b["max_abs_err"])}


def assert_parity(stats: dict, what: str = "") -> None:
    assert stats["violations"] == 0, (what, stats)
