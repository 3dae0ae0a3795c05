"""CPU oracle for packed variable-length QK-RoPE (test infrastructure only).

This package is the plain, slow definition the CUDA library is checked against.
Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
and reference arms may import it; the product path never does.  It shares no code
with the CUDA library: its arithmetic lives in ``rope_oracle.c`` (plain C, built
with ``-ffp-contract=off``), and this module only marshals numpy arrays.

What each function follows (restated, not copied):

* ``positions`` -- unsloth.ai "3x faster training with packing", section
  "Packing non contaminé": position ids restart at each packed-sample boundary.
* ``inv_freq`` / ``cos_sin`` -- rotary base ``rope_theta`` as named in the TRL
  "training beyond 1M tokens" page, YaRN section; the RoFormer frequency form is a
  reading (the pages print no formula).  ``scale`` is that section's linear position
  rescale ("position 100 000 becomes 25 000" with factor 4).
* ``rope_rows`` / ``rope_packed`` -- unsloth.ai page, section "Kernel Triton QK
  RoPE fusionné avec packing": ``x*cos + rotate_half(x)*sin``; backward is the same
  with sin negated (``R^T``).
* ``glu_fwd`` / ``glu_bwd`` (``glu_oracle.c``) -- the SwiGLU / GeGLU kernels of the
  same page (updated for int64 indexing) and the MLP line
  ``down_proj(act_fn(gate_proj(x)) * up_proj(x))`` of the TRL page, in binary64,
  rounded once to bf16.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "rope_oracle.c")
SOURCES = [SOURCE, os.path.join(_HERE, "glu_oracle.c")]
LIB_PATH = os.path.join(_HERE, "librope_oracle.so")
CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-shared", "-fPIC"]


def compile_source(src, out: str) -> str:
    """Compile oracle C sources (one path or a list) into a shared library, no FMA
    contraction."""
    srcs = [src] if isinstance(src, str) else list(src)
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", *CFLAGS, *srcs, "-o", tmp, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle if its library is missing or older than a source."""
    if force or not os.path.exists(LIB_PATH) or \
            any(os.path.getmtime(LIB_PATH) < os.path.getmtime(p) for p in SOURCES):
        compile_source(SOURCES, LIB_PATH)
    return LIB_PATH


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class Oracle:
    """ctypes view of one compiled oracle library (the default one, or a test build)."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        i32p = ctypes.POINTER(ctypes.c_int32)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        f32p = ctypes.POINTER(ctypes.c_float)
        lib.oracle_positions.argtypes = [i32p, ctypes.c_int32, ctypes.c_int64, i32p]
        lib.oracle_positions.restype = ctypes.c_int
        lib.oracle_inv_freq.argtypes = [ctypes.c_double, ctypes.c_int32, f32p]
        lib.oracle_inv_freq.restype = None
        lib.oracle_cos_sin.argtypes = [ctypes.c_int32, ctypes.c_double, ctypes.c_int32, f32p, f32p]
        lib.oracle_cos_sin.restype = None
        lib.oracle_rope_rows.argtypes = [u16p, u16p, ctypes.c_int64, i32p, ctypes.c_int32,
                                         ctypes.c_int32, ctypes.c_double, ctypes.c_int32]
        lib.oracle_rope_rows.restype = None
        lib.oracle_rope_packed.argtypes = [u16p, u16p, i32p, ctypes.c_int32, ctypes.c_int64,
                                           ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                           ctypes.c_int32, i32p]
        lib.oracle_rope_packed.restype = ctypes.c_int
        lib.oracle_inv_freq_scaled.argtypes = [ctypes.c_double, ctypes.c_int32, ctypes.c_double, f32p]
        lib.oracle_inv_freq_scaled.restype = None
        lib.oracle_cos_sin_scaled.argtypes = [ctypes.c_int32, ctypes.c_double, ctypes.c_int32, ctypes.c_double,
                                              f32p, f32p]
        lib.oracle_cos_sin_scaled.restype = None
        lib.oracle_rope_rows_scaled.argtypes = [u16p, u16p, ctypes.c_int64, i32p, ctypes.c_int32,
                                                ctypes.c_int32, ctypes.c_double, ctypes.c_double,
                                                ctypes.c_int32]
        lib.oracle_rope_rows_scaled.restype = None
        lib.oracle_glu_activation.argtypes = [ctypes.c_int32, ctypes.c_double,
                                              ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
        lib.oracle_glu_activation.restype = None
        lib.oracle_glu_fwd.argtypes = [ctypes.c_int32, u16p, u16p, u16p, ctypes.c_int64]
        lib.oracle_glu_fwd.restype = None
        lib.oracle_glu_bwd.argtypes = [ctypes.c_int32, u16p, u16p, u16p, u16p, u16p, ctypes.c_int64]
        lib.oracle_glu_bwd.restype = None
        lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_double_to_bf16.restype = ctypes.c_uint16
        lib.oracle_float_to_bf16.argtypes = [ctypes.c_float]
        lib.oracle_float_to_bf16.restype = ctypes.c_uint16
        self.lib = lib
        self.path = lib_path

    def positions(self, cu_seqlens, total_tokens: int) -> np.ndarray:
        """int32 position of every token in its packed sample; -1 outside every sample."""
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        out = np.empty(int(total_tokens), dtype=np.int32)
        rc = self.lib.oracle_positions(_ptr(cu, ctypes.c_int32), cu.size - 1, int(total_tokens),
                                       _ptr(out, ctypes.c_int32))
        if rc != 0:
            raise ValueError("cu_seqlens is not non-decreasing within [0, total_tokens]")
        return out

    def inv_freq(self, theta: float, head_dim: int, scale: float = 1.0) -> np.ndarray:
        w = np.empty(head_dim // 2, dtype=np.float32)
        self.lib.oracle_inv_freq_scaled(float(theta), int(head_dim), float(scale), _ptr(w, ctypes.c_float))
        return w

    def cos_sin(self, pos: int, theta: float, head_dim: int, scale: float = 1.0):
        """(c, s) float32 arrays of length head_dim/2 for one position."""
        c = np.empty(head_dim // 2, dtype=np.float32)
        s = np.empty(head_dim // 2, dtype=np.float32)
        self.lib.oracle_cos_sin_scaled(int(pos), float(theta), int(head_dim), float(scale),
                                       _ptr(c, ctypes.c_float), _ptr(s, ctypes.c_float))
        return c, s

    def rope_rows(self, x_bits: np.ndarray, pos, theta: float, bwd: bool = False,
                  scale: float = 1.0) -> np.ndarray:
        """Rotate token rows.  x_bits: uint16 bf16 bit patterns [rows, H, d]; pos: int32
        [rows] (-1 leaves a row unchanged); scale: linear position rescale (1 = none).
        Returns a new uint16 array."""
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        rows, H, d = x.shape
        p = np.ascontiguousarray(pos, dtype=np.int32)
        assert p.shape == (rows,) and d % 2 == 0 and d <= 1024
        y = np.empty_like(x)
        self.lib.oracle_rope_rows_scaled(_ptr(x, ctypes.c_uint16), _ptr(y, ctypes.c_uint16), rows,
                                         _ptr(p, ctypes.c_int32), H, d, float(theta), float(scale),
                                         1 if bwd else 0)
        return y

    def rope_packed(self, x_bits: np.ndarray, cu_seqlens, theta: float, bwd: bool = False) -> np.ndarray:
        """Whole packed tensor [T, H, d] (uint16 bf16 bits), positions from cu_seqlens."""
        x = np.ascontiguousarray(x_bits, dtype=np.uint16)
        T, H, d = x.shape
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        y = np.empty_like(x)
        scratch = np.empty(T, dtype=np.int32)
        rc = self.lib.oracle_rope_packed(_ptr(x, ctypes.c_uint16), _ptr(y, ctypes.c_uint16),
                                         _ptr(cu, ctypes.c_int32), cu.size - 1, T, H, d,
                                         float(theta), 1 if bwd else 0,
                                         _ptr(scratch, ctypes.c_int32))
        if rc != 0:
            raise ValueError("cu_seqlens is not non-decreasing within [0, total_tokens]")
        return y

    def float_to_bf16_bits(self, v: float) -> int:
        return int(self.lib.oracle_float_to_bf16(float(v)))

    # ---- gated MLP activations (glu_oracle.c)
    GLU_KINDS = {"swiglu": 0, "geglu": 1, "geglu_tanh": 2}

    def glu_activation(self, kind: str, x: float):
        """(act(x), act'(x)) in binary64."""
        a, da = ctypes.c_double(), ctypes.c_double()
        self.lib.oracle_glu_activation(self.GLU_KINDS[kind], float(x), ctypes.byref(a), ctypes.byref(da))
        return a.value, da.value

    def glu_fwd(self, kind: str, e_bits, g_bits):
        """h = bf16(act(e) * g), elementwise on uint16 bf16 bit arrays of one shape."""
        e = np.ascontiguousarray(e_bits, dtype=np.uint16)
        g = np.ascontiguousarray(g_bits, dtype=np.uint16)
        assert e.shape == g.shape
        h = np.empty_like(e)
        self.lib.oracle_glu_fwd(self.GLU_KINDS[kind], _ptr(e, ctypes.c_uint16), _ptr(g, ctypes.c_uint16),
                                _ptr(h, ctypes.c_uint16), e.size)
        return h

    def glu_bwd(self, kind: str, dh_bits, e_bits, g_bits):
        """(de, dg) = (bf16(dh * g * act'(e)), bf16(dh * act(e)))."""
        dh = np.ascontiguousarray(dh_bits, dtype=np.uint16)
        e = np.ascontiguousarray(e_bits, dtype=np.uint16)
        g = np.ascontiguousarray(g_bits, dtype=np.uint16)
        assert dh.shape == e.shape == g.shape
        de = np.empty_like(e)
        dg = np.empty_like(e)
        self.lib.oracle_glu_bwd(self.GLU_KINDS[kind], _ptr(dh, ctypes.c_uint16), _ptr(e, ctypes.c_uint16),
                                _ptr(g, ctypes.c_uint16), _ptr(de, ctypes.c_uint16), _ptr(dg, ctypes.c_uint16),
                                e.size)
        return de, dg

    def double_to_bf16_bits(self, v: float) -> int:
        return int(self.lib.oracle_double_to_bf16(float(v)))


_default = None


def get() -> Oracle:
    """The oracle built from ``rope_oracle.c`` (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def positions(cu_seqlens, total_tokens):
    return get().positions(cu_seqlens, total_tokens)


def inv_freq(theta, head_dim, scale=1.0):
    return get().inv_freq(theta, head_dim, scale)


def cos_sin(pos, theta, head_dim, scale=1.0):
    return get().cos_sin(pos, theta, head_dim, scale)


def rope_rows(x_bits, pos, theta, bwd=False, scale=1.0):
    return get().rope_rows(x_bits, pos, theta, bwd, scale)


def rope_packed(x_bits, cu_seqlens, theta, bwd=False):
    return get().rope_packed(x_bits, cu_seqlens, theta, bwd)


def float_to_bf16_bits(v):
    return get().float_to_bf16_bits(v)


def glu_fwd(kind, e_bits, g_bits):
    return get().glu_fwd(kind, e_bits, g_bits)


def glu_bwd(kind, dh_bits, e_bits, g_bits):
    return get().glu_bwd(kind, dh_bits, e_bits, g_bits)
