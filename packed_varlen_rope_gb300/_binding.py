"""ctypes binding of librope_qk.so: argument marshalling only.

Every function here has the name of the C entry point it calls and does no arithmetic
of the method: it checks tensor dtypes/devices, turns tensors into pointers and the
current torch stream into a ``cudaStream_t``, and raises ``RopeError`` on a non-zero
status.  There is no fallback: if the library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "librope_qk.so")

EXPORTS = (
    "rope_qk_fwd", "rope_qk_bwd", "rope_qk_apply", "rope_cos_sin_cache_build",
    "rope_cos_sin_cache_bytes", "rope_qk_positions",
    "rope_validate_cu_seqlens", "rope_qk_inv_freq", "rope_strerror", "rope_qk_abi_version",
    "glu_fwd", "glu_bwd", "rope_qk_host", "rope_qk_host_static", "rope_qk_launch_info",
    "rope_cos_sin_eval",
)

GLU_KINDS = {"swiglu": 0, "geglu": 1, "geglu_tanh": 2}

ROPE_CU_NEGATIVE_START = 0x1
ROPE_CU_DECREASING = 0x2
ROPE_CU_PAST_END = 0x4
ROPE_CU_NONZERO_START = 0x8
ROPE_FLAG_POSITION_IDS_INT64 = 0x1
ROPE_MAX_SEGMENTS = 16

_lib = None


class RopeCosSinCacheDesc(ctypes.Structure):
    """Mirror of ``rope_cos_sin_cache`` in include/rope_qk.h (written by the library's
    cache build only)."""

    _fields_ = [
        ("data", ctypes.c_void_p), ("rows", ctypes.c_int64), ("head_dim", ctypes.c_int32),
        ("device", ctypes.c_int32), ("theta", ctypes.c_double), ("position_scale", ctypes.c_double),
        ("check", ctypes.c_uint64),
    ]


class RopeQKSegment(ctypes.Structure):
    """Mirror of ``rope_qk_segment``: rows from ``row_start`` on are tokens
    ``token_start``, ``token_start + 1``, ... of cu_seqlens' stream."""

    _fields_ = [("row_start", ctypes.c_int64), ("token_start", ctypes.c_int64)]


class RopeQKDesc(ctypes.Structure):
    """Mirror of ``rope_qk_desc`` in include/rope_qk.h (same field order and types)."""

    _fields_ = [
        ("q", ctypes.c_void_p), ("q_stride_token", ctypes.c_int64), ("q_stride_head", ctypes.c_int64),
        ("k", ctypes.c_void_p), ("k_stride_token", ctypes.c_int64), ("k_stride_head", ctypes.c_int64),
        ("q_out", ctypes.c_void_p), ("q_out_stride_token", ctypes.c_int64), ("q_out_stride_head", ctypes.c_int64),
        ("k_out", ctypes.c_void_p), ("k_out_stride_token", ctypes.c_int64), ("k_out_stride_head", ctypes.c_int64),
        ("cu_seqlens", ctypes.c_void_p), ("n_seqs", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("position_ids", ctypes.c_void_p), ("total_tokens", ctypes.c_int64), ("token_offset", ctypes.c_int64),
        ("theta", ctypes.c_double), ("position_scale", ctypes.c_double),
        ("cos_sin_cache", ctypes.POINTER(RopeCosSinCacheDesc)),
        ("backward", ctypes.c_int32), ("flags", ctypes.c_int32),
        ("seq_used", ctypes.c_void_p),
        ("segments", ctypes.POINTER(RopeQKSegment)), ("n_segments", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]


class RopeQKLaunch(ctypes.Structure):
    """Mirror of ``rope_qk_launch``: what rope_qk_apply launches for a descriptor."""

    _fields_ = [("head_dim_instance", ctypes.c_int32), ("long_index", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("tile_tokens", ctypes.c_int32), ("threads", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
                ("unroll", ctypes.c_int32)]

    def kernel_name(self) -> str:
        """The rotation kernel's instance as its template reads: rope_qk_tile_kernel<D, LONG, U>."""
        return "rope_qk_tile_kernel<%d,%s,%d>" % (self.head_dim_instance, "true" if self.long_index else "false",
                                                  self.unroll)


class CosSinCache:
    """A cos/sin cache: the device table ``data`` (float32 [rows, 4, head_dim/16, 4])
    and the descriptor the library's build wrote for it, which records the theta,
    head_dim, position_scale and device it serves.  Passed as ``cos_sin_cache=`` to the
    rotations; the library rejects it for any other theta, head_dim, scale or device."""

    def __init__(self, data, desc: RopeCosSinCacheDesc):
        self.data = data
        self.desc = desc

    @property
    def rows(self) -> int:
        return int(self.desc.rows)

    @property
    def head_dim(self) -> int:
        return int(self.desc.head_dim)

    @property
    def theta(self) -> float:
        return float(self.desc.theta)

    @property
    def position_scale(self) -> float:
        return float(self.desc.position_scale)

    @property
    def device(self):
        return self.data.device

    def ref(self):
        """``rope_cos_sin_cache *`` for a C call."""
        return ctypes.pointer(self.desc)


class RopeError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__("%s failed with status %d: %s" % (fn, status, text))
        self.status = status


def load_library(path: Optional[str] = None):
    """Load librope_qk.so (built by ``packed_varlen_rope_gb300.build``) and declare its
    signatures.  Raises ``OSError`` when the library has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise OSError("librope_qk.so is not built (%s); run packed_varlen_rope_gb300.build.build()" % p)
    lib = ctypes.CDLL(p)
    vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    cache_p = ctypes.POINTER(RopeCosSinCacheDesc)
    rope_args = [vp, vp, vp, i32, i64, i32, i32, i32, dbl, i32, vp, vp, cache_p, vp]
    for name in ("rope_qk_fwd", "rope_qk_bwd"):
        getattr(lib, name).argtypes = rope_args
        getattr(lib, name).restype = ctypes.c_int
    lib.rope_qk_apply.argtypes = [ctypes.POINTER(RopeQKDesc), vp]
    lib.rope_qk_apply.restype = ctypes.c_int
    lib.rope_qk_launch_info.argtypes = [ctypes.POINTER(RopeQKDesc), ctypes.POINTER(RopeQKLaunch)]
    lib.rope_qk_launch_info.restype = ctypes.c_int
    lib.rope_qk_host.argtypes = [ctypes.POINTER(RopeQKDesc), vp, i64, vp]
    lib.rope_qk_host.restype = ctypes.c_int
    lib.rope_qk_host_static.argtypes = [ctypes.POINTER(RopeQKDesc), vp]
    lib.rope_qk_host_static.restype = ctypes.c_int
    lib.rope_cos_sin_cache_build.argtypes = [cache_p, vp, i64, i32, dbl, dbl, vp]
    lib.rope_cos_sin_cache_build.restype = ctypes.c_int
    lib.rope_cos_sin_cache_bytes.argtypes = [i64, i32]
    lib.rope_cos_sin_cache_bytes.restype = ctypes.c_int64
    lib.rope_qk_positions.argtypes = [vp, i32, i64, vp, vp]
    lib.rope_qk_positions.restype = ctypes.c_int
    lib.rope_validate_cu_seqlens.argtypes = [vp, i32, i64, vp, vp]
    lib.rope_validate_cu_seqlens.restype = ctypes.c_int
    lib.rope_cos_sin_eval.argtypes = [vp, vp, vp, i64, i32, vp]
    lib.rope_cos_sin_eval.restype = ctypes.c_int
    lib.rope_qk_inv_freq.argtypes = [dbl, i32, dbl, ctypes.POINTER(ctypes.c_float)]
    lib.rope_qk_inv_freq.restype = ctypes.c_int
    lib.rope_strerror.argtypes = [ctypes.c_int]
    lib.rope_strerror.restype = ctypes.c_char_p
    lib.glu_fwd.argtypes = [i32, vp, i64, vp, i64, vp, i64, i64, i64, vp]
    lib.glu_fwd.restype = ctypes.c_int
    lib.glu_bwd.argtypes = [i32, vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, i64, i64, vp]
    lib.glu_bwd.restype = ctypes.c_int
    lib.rope_qk_abi_version.argtypes = []
    lib.rope_qk_abi_version.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def rope_strerror(status: int) -> str:
    return load_library().rope_strerror(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise RopeError(fn, status, rope_strerror(status))


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def _stream(stream, device) -> int:
    """Raw cudaStream_t of ``stream`` (a torch stream or an int), else the current stream
    of ``device``."""
    import torch

    if stream is None:
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            return int(raw(device.index if device.index is not None else torch.cuda.current_device()))
        return int(torch.cuda.current_stream(device).cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _on(device, fn, *args):
    """Call library entry point ``fn`` with ``device`` current: the library launches on
    the calling thread's current device, and the stream passed belongs to ``device``.
    The device is switched (and restored) only when another one is current."""
    import torch

    if device.index is None or device.index == torch.cuda.current_device():
        return fn(*args)
    with torch.cuda.device(device):
        return fn(*args)


def _check_qk(q, k):
    import torch

    for name, t in (("q", q), ("k", k)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 3:
            raise ValueError("%s must be a contiguous CUDA bf16 tensor [tokens, heads, head_dim]" % name)
    if q.shape[0] != k.shape[0] or q.shape[2] != k.shape[2] or q.device != k.device:
        raise ValueError("q and k must share tokens, head_dim and device")


def _check_cu(cu_seqlens, device):
    import torch

    if cu_seqlens.dtype != torch.int32 or cu_seqlens.device != device or not cu_seqlens.is_contiguous():
        raise ValueError("cu_seqlens must be a contiguous int32 tensor on the device of q")


def _cache_arg(cache, head_dim: int, device):
    """``rope_cos_sin_cache *`` of a ``CosSinCache`` (None: a NULL pointer) after the
    checks the C side cannot make on a tensor: type, dtype, layout and device.  theta,
    head_dim and position_scale are checked by the library against its descriptor."""
    import torch

    if cache is None:
        return None
    if not isinstance(cache, CosSinCache):
        raise ValueError("cos_sin_cache must be a CosSinCache (new_cos_sin_cache / rope_cos_sin_cache_build)")
    t = cache.data
    if t.dtype != torch.float32:
        raise ValueError("cos_sin_cache must hold float32 values, not %s" % t.dtype)
    if t.dim() != 4 or tuple(t.shape[1:]) != (4, head_dim // 16, 4) or t.shape[0] != cache.rows or \
            not t.is_contiguous():
        raise ValueError("cos_sin_cache must hold a contiguous [rows, 4, head_dim/16, 4] table for head_dim %d, "
                         "got %s" % (head_dim, tuple(t.shape)))
    if not t.is_cuda or t.device != device:
        raise ValueError("cos_sin_cache is on %s, the rotation runs on %s" % (t.device, device))
    if cache.rows and cache.desc.data != t.data_ptr():
        raise ValueError("cos_sin_cache's descriptor does not describe its tensor")
    return cache.ref()


def _rope(fn_name, q, k, cu_seqlens, theta, in_place, q_out, k_out, cos_sin_cache, stream):
    _check_qk(q, k)
    _check_cu(cu_seqlens, q.device)
    T, hq, d = q.shape
    hkv = k.shape[1]
    if not in_place:
        if q_out is None or k_out is None:
            raise ValueError("q_out and k_out are required when in_place is False")
        _check_qk(q_out, k_out)
        if q_out.shape != q.shape or k_out.shape != k.shape or q_out.device != q.device:
            raise ValueError("q_out/k_out must have the shapes and device of q/k")
    cache = _cache_arg(cos_sin_cache, d, q.device)
    fn = getattr(load_library(), fn_name)
    st = _on(q.device, fn, _ptr(q), _ptr(k), _ptr(cu_seqlens), cu_seqlens.numel() - 1, T, hq, hkv, d,
             float(theta), 1 if in_place else 0, _ptr(q_out) if not in_place else None,
             _ptr(k_out) if not in_place else None, cache, _stream(stream, q.device))
    _check(fn_name, st)
    return (q, k) if in_place else (q_out, k_out)


def rope_qk_fwd(q, k, cu_seqlens, theta: float, in_place: bool = True, q_out=None, k_out=None,
                cos_sin_cache=None, stream=None):
    """Rotate Q [T, Hq, d] and K [T, Hkv, d] (bf16, CUDA) by their packed positions.
    ``cos_sin_cache``: an optional ``CosSinCache`` built for the same theta and head_dim.
    Returns (q, k) in place, else (q_out, k_out)."""
    return _rope("rope_qk_fwd", q, k, cu_seqlens, theta, in_place, q_out, k_out, cos_sin_cache, stream)


def rope_qk_bwd(q, k, cu_seqlens, theta: float, in_place: bool = True, q_out=None, k_out=None,
                cos_sin_cache=None, stream=None):
    """Transpose rotation (sin negated): q and k hold the gradients dL/dY of Q and K and
    receive dL/dX (or q_out/k_out do).  Same arguments as ``rope_qk_fwd``."""
    return _rope("rope_qk_bwd", q, k, cu_seqlens, theta, in_place, q_out, k_out, cos_sin_cache, stream)


def rope_cos_sin_cache_build(data, theta: float, stream=None, position_scale: float = 1.0) -> CosSinCache:
    """Fill a float32 [rows, 4, head_dim/16, 4] CUDA tensor with (cos, sin) per position
    (entry [p, q, c] = c_j, s_j, c_j+1, s_j+1 for j = 8c + 2q) for one theta and linear
    position_scale, and return it as a ``CosSinCache`` with the library's descriptor."""
    import torch

    if data.dtype != torch.float32 or not data.is_cuda or not data.is_contiguous() or \
            data.dim() != 4 or data.shape[1] != 4 or data.shape[3] != 4:
        raise ValueError("cache must be a contiguous CUDA float32 [rows, 4, head_dim/16, 4] tensor")
    desc = RopeCosSinCacheDesc()
    st = _on(data.device, load_library().rope_cos_sin_cache_build, ctypes.byref(desc), _ptr(data), data.shape[0],
             16 * data.shape[2], float(theta), float(position_scale), _stream(stream, data.device))
    _check("rope_cos_sin_cache_build", st)
    return CosSinCache(data, desc)


def new_cos_sin_cache(rows: int, head_dim: int, theta: float, device="cuda", stream=None,
                      position_scale: float = 1.0) -> CosSinCache:
    """Allocate (through torch) and build a cos/sin cache of ``rows`` positions."""
    import torch

    data = torch.empty((rows, 4, head_dim // 16, 4), dtype=torch.float32, device=device)
    return rope_cos_sin_cache_build(data, theta, stream, position_scale)


def cache_as_cos_sin(cache_np):
    """View a cache table copied to the host (numpy [rows, 4, d/16, 4]) as [rows, d/2, 2]
    (c, s)."""
    rows, _, cph, _ = cache_np.shape
    return cache_np.transpose(0, 2, 1, 3).reshape(rows, 8 * cph, 2)


def rope_qk_positions(cu_seqlens, total_tokens: int, pos_out=None, stream=None):
    """int32 [total_tokens] positions exactly as the kernels derive them (-1 outside)."""
    import torch

    if pos_out is None:
        pos_out = torch.empty(int(total_tokens), dtype=torch.int32, device=cu_seqlens.device)
    _check_cu(cu_seqlens, pos_out.device)
    st = _on(cu_seqlens.device, load_library().rope_qk_positions, _ptr(cu_seqlens), cu_seqlens.numel() - 1,
             int(total_tokens), _ptr(pos_out), _stream(stream, cu_seqlens.device))
    _check("rope_qk_positions", st)
    return pos_out


def rope_validate_cu_seqlens(cu_seqlens, total_tokens: int, err_word=None, stream=None):
    """Device check of cu_seqlens; returns the int32 [1] device word of ROPE_CU_* bits."""
    import torch

    if err_word is None:
        err_word = torch.empty(1, dtype=torch.int32, device=cu_seqlens.device)
    st = _on(cu_seqlens.device, load_library().rope_validate_cu_seqlens, _ptr(cu_seqlens),
             cu_seqlens.numel() - 1, int(total_tokens), _ptr(err_word), _stream(stream, cu_seqlens.device))
    _check("rope_validate_cu_seqlens", st)
    return err_word


COS_SIN_MODES = {"as_rotation": 0, "binary64": 1, "binary32_only": 2}


def rope_cos_sin_eval(phi, mode: str = "as_rotation", stream=None):
    """(cos, sin) float32 CUDA tensors of the float32 CUDA angles ``phi`` as the rotation
    evaluates them ("as_rotation"), in binary64 only ("binary64"), or in binary32 only
    with NaN where that evaluation leaves the rounding to binary64 ("binary32_only")."""
    import torch

    if phi.dtype != torch.float32 or not phi.is_cuda or not phi.is_contiguous():
        raise ValueError("phi must be a contiguous float32 CUDA tensor")
    c, s = torch.empty_like(phi), torch.empty_like(phi)
    st = _on(phi.device, load_library().rope_cos_sin_eval, _ptr(phi), _ptr(c), _ptr(s), phi.numel(),
             COS_SIN_MODES[mode], _stream(stream, phi.device))
    _check("rope_cos_sin_eval", st)
    return c, s


def rope_qk_inv_freq(theta: float, head_dim: int, position_scale: float = 1.0):
    """Host-side inverse frequencies (numpy float32 [head_dim/2]) as the kernels use them."""
    import numpy as np

    w = np.empty(int(head_dim) // 2, dtype=np.float32)
    st = load_library().rope_qk_inv_freq(float(theta), int(head_dim), float(position_scale),
                                         w.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    _check("rope_qk_inv_freq", st)
    return w


def _view_args(t, name):
    import torch

    if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 3 or t.stride(2) != 1:
        raise ValueError("%s must be a CUDA bf16 [tokens, heads, head_dim] view with head_dim contiguous" % name)
    return _ptr(t), t.stride(0), t.stride(1)


def _segments_arg(segments, T: int):
    """(ctypes array, count) of a list of (row_start, token_start) pairs."""
    if segments is None:
        return None, 0
    segs = [(int(a), int(b)) for a, b in segments]
    if not 1 <= len(segs) <= ROPE_MAX_SEGMENTS:
        raise ValueError("give 1 to %d segments" % ROPE_MAX_SEGMENTS)
    arr = (RopeQKSegment * len(segs))(*[RopeQKSegment(a, b) for a, b in segs])
    return arr, len(segs)


def _apply_desc(q, k, theta, cu_seqlens, position_ids, backward, q_out, k_out, token_offset, position_scale,
                cos_sin_cache, seq_used, segments):
    """The descriptor of a rope_qk_apply call (and the objects it points into, which must
    outlive the call)."""
    qp, q_ts, q_hs = _view_args(q, "q")
    kp, k_ts, k_hs = _view_args(k, "k")
    if q.shape[0] != k.shape[0] or q.shape[2] != k.shape[2] or q.device != k.device:
        raise ValueError("q and k must share tokens, head_dim and device")
    T, hq, d = q.shape
    desc = RopeQKDesc()
    desc.q, desc.q_stride_token, desc.q_stride_head = qp, q_ts, q_hs
    desc.k, desc.k_stride_token, desc.k_stride_head = kp, k_ts, k_hs
    if (q_out is None) != (k_out is None):
        raise ValueError("give both q_out and k_out, or neither (in place)")
    if q_out is not None:
        if q_out.shape != q.shape or k_out.shape != k.shape or q_out.device != q.device or \
                k_out.device != q.device:
            raise ValueError("q_out/k_out must have the shapes and device of q/k")
        desc.q_out, desc.q_out_stride_token, desc.q_out_stride_head = _view_args(q_out, "q_out")
        desc.k_out, desc.k_out_stride_token, desc.k_out_stride_head = _view_args(k_out, "k_out")
    _positions_args(desc, T, q.device, cu_seqlens, position_ids, seq_used)
    seg_arr, desc.n_segments = _segments_arg(segments, T)
    if seg_arr is not None:
        desc.segments = seg_arr
    desc.n_q_heads, desc.n_kv_heads, desc.head_dim = hq, k.shape[1], d
    desc.total_tokens = T
    desc.token_offset = int(token_offset)
    desc.theta = float(theta)
    desc.position_scale = float(position_scale)
    cache = _cache_arg(cos_sin_cache, d, q.device)
    if cache is not None:
        desc.cos_sin_cache = cache
    desc.backward = 1 if backward else 0
    return desc, (seg_arr, cache)


def rope_qk_apply(q, k, theta: float, cu_seqlens=None, position_ids=None, backward: bool = False,
                  q_out=None, k_out=None, token_offset: int = 0, position_scale: float = 1.0,
                  cos_sin_cache=None, stream=None, seq_used=None, segments=None):
    """General form of the rotation (C entry point ``rope_qk_apply``).

    q, k: bf16 CUDA views [T, Hq, d] and [T, Hkv, d] with any token/head strides
    (head_dim contiguous) -- e.g. the Q and K slices of one fused QKV output, rotated in
    place.  Positions come from ``position_ids`` (int32 or int64 [T]) if given, else from
    ``cu_seqlens`` with row r read as token ``token_offset + r`` (and, with
    ``seq_used``, only the first seq_used[s] tokens of sample s rotated).  ``segments``:
    a list of (row_start, token_start) pairs, rows from row_start on being tokens
    token_start, token_start + 1, ... (a context-parallel rank's non-adjacent shards in
    one call; see ``cp_shards``).  ``position_scale`` is the linear position rescale
    (1 = none).  Returns (q, k) in place, else (q_out, k_out)."""
    desc, keep = _apply_desc(q, k, theta, cu_seqlens, position_ids, backward, q_out, k_out, token_offset,
                             position_scale, cos_sin_cache, seq_used, segments)
    st = _on(q.device, load_library().rope_qk_apply, ctypes.byref(desc), _stream(stream, q.device))
    del keep
    _check("rope_qk_apply", st)
    return (q, k) if q_out is None else (q_out, k_out)


def rope_qk_launch_info(q, k, theta: float, cu_seqlens=None, position_ids=None, backward: bool = False,
                        q_out=None, k_out=None, token_offset: int = 0, position_scale: float = 1.0,
                        cos_sin_cache=None, seq_used=None, segments=None) -> RopeQKLaunch:
    """What ``rope_qk_apply`` with the same arguments would launch (C entry point
    ``rope_qk_launch_info``; no launch, no CUDA call): ``.kernel_name()``, grid, tile."""
    desc, keep = _apply_desc(q, k, theta, cu_seqlens, position_ids, backward, q_out, k_out, token_offset,
                             position_scale, cos_sin_cache, seq_used, segments)
    info = RopeQKLaunch()
    st = load_library().rope_qk_launch_info(ctypes.byref(desc), ctypes.byref(info))
    del keep
    _check("rope_qk_launch_info", st)
    return info


def _positions_args(desc, T: int, device, cu_seqlens, position_ids, seq_used):
    """Fill the position source of a descriptor: int32/int64 position ids, or cu_seqlens
    (with seq_used), all contiguous tensors on ``device``."""
    import torch

    if position_ids is not None:
        if position_ids.dtype not in (torch.int32, torch.int64) or position_ids.device != device or \
                not position_ids.is_contiguous() or position_ids.numel() != T:
            raise ValueError("position_ids must be a contiguous int32 or int64 [tokens] tensor on %s" % device)
        desc.position_ids = _ptr(position_ids)
        if position_ids.dtype == torch.int64:
            desc.flags |= ROPE_FLAG_POSITION_IDS_INT64
    elif cu_seqlens is not None:
        _check_cu(cu_seqlens, device)
        desc.cu_seqlens = _ptr(cu_seqlens)
        desc.n_seqs = cu_seqlens.numel() - 1
        if seq_used is not None:
            _check_cu(seq_used, device)
            if seq_used.numel() != desc.n_seqs:
                raise ValueError("seq_used must hold one int32 per sample")
            desc.seq_used = _ptr(seq_used)
    else:
        raise ValueError("give cu_seqlens or position_ids")


def rope_qk_abi_version() -> int:
    return int(load_library().rope_qk_abi_version())


def _mat_args(t, name, shape, device):
    import torch

    if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 2 or (t.numel() and t.stride(1) != 1):
        raise ValueError("%s must be a CUDA bf16 [rows, cols] view with contiguous rows" % name)
    if t.device != device:
        raise ValueError("%s must be on %s" % (name, device))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s" % (name, tuple(shape)))
    return _ptr(t), t.stride(0)


def glu_fwd(kind: str, e, g, h=None, stream=None):
    """h = act(e) * g for SwiGLU ("swiglu") or GeGLU ("geglu", "geglu_tanh").  e, g, h:
    bf16 [rows, cols] CUDA views (cols a multiple of 8); h may be e or g (in place).
    Returns h (a new tensor when not given)."""
    import torch

    shape = tuple(e.shape)
    if h is None:
        h = torch.empty(shape, dtype=torch.bfloat16, device=e.device)
    ep, es = _mat_args(e, "e", shape, e.device)
    gp, gs = _mat_args(g, "g", shape, e.device)
    hp, hs = _mat_args(h, "h", shape, e.device)
    st = _on(e.device, load_library().glu_fwd, GLU_KINDS[kind], ep, es, gp, gs, hp, hs, shape[0], shape[1],
             _stream(stream, e.device))
    _check("glu_fwd", st)
    return h


def glu_bwd(kind: str, dh, e, g, de=None, dg=None, stream=None):
    """de = dh * g * act'(e), dg = dh * act(e).  de/dg may be e/g (or dh) for an
    in-place backward.  Returns (de, dg)."""
    import torch

    shape = tuple(e.shape)
    if de is None:
        de = torch.empty(shape, dtype=torch.bfloat16, device=e.device)
    if dg is None:
        dg = torch.empty(shape, dtype=torch.bfloat16, device=e.device)
    args = []
    for name, t in (("dh", dh), ("e", e), ("g", g), ("de", de), ("dg", dg)):
        args += list(_mat_args(t, name, shape, e.device))
    st = _on(e.device, load_library().glu_bwd, GLU_KINDS[kind], *args, shape[0], shape[1],
             _stream(stream, e.device))
    _check("glu_bwd", st)
    return de, dg


def rope_qk_host(q, k, theta: float, workspace=None, cu_seqlens=None, position_ids=None, backward: bool = False,
                 q_out=None, k_out=None, token_offset: int = 0, position_scale: float = 1.0,
                 cos_sin_cache=None, stream=None, device=None, seq_used=None, segments=None):
    """Rotate Q [T, Hq, d] and K [T, Hkv, d] that live in HOST memory (contiguous bf16 CPU
    tensors, pinned for overlapped copies), streaming them through ``workspace`` (a
    CUDA tensor of any dtype used as raw staging memory).  Without a workspace the
    library's built-in 32 MiB staging array is used and nothing is allocated
    (``rope_qk_host_static``; ``device`` then names the GPU).  cu_seqlens /
    position_ids / seq_used (with cu_seqlens: the used tokens of each sample of a
    padded batch) are CUDA tensors; cos_sin_cache a ``CosSinCache`` on the same GPU;
    segments as for ``rope_qk_apply``.  q_out and k_out, if given, are host tensors of
    exactly q's and k's shapes.  Asynchronous on ``stream``: synchronise it before
    reading the results.  Returns (q, k) or (q_out, k_out)."""
    import torch

    for name, t in (("q", q), ("k", k), ("q_out", q_out), ("k_out", k_out)):
        if t is None:
            continue
        if t.dtype != torch.bfloat16 or t.is_cuda or not t.is_contiguous() or t.dim() != 3:
            raise ValueError("%s must be a contiguous host (CPU) bf16 tensor [tokens, heads, head_dim]" % name)
    if q.shape[0] != k.shape[0] or q.shape[2] != k.shape[2]:
        raise ValueError("q and k must share tokens and head_dim")
    if (q_out is None) != (k_out is None):
        raise ValueError("give both q_out and k_out, or neither")
    if q_out is not None and (q_out.shape != q.shape or k_out.shape != k.shape):
        raise ValueError("q_out and k_out must have exactly the shapes of q and k")
    if workspace is not None and (not workspace.is_cuda or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    T, hq, d = q.shape
    if workspace is not None:
        dev = workspace.device
    elif device is not None:
        dev = torch.device(device)
    else:
        dev = torch.device("cuda", torch.cuda.current_device())
    if dev.type != "cuda":
        raise ValueError("the staging device must be a CUDA device")
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    cache = _cache_arg(cos_sin_cache, d, dev)
    desc = RopeQKDesc()
    desc.q, desc.q_stride_token, desc.q_stride_head = _ptr(q), hq * d, d
    desc.k, desc.k_stride_token, desc.k_stride_head = _ptr(k), k.shape[1] * d, d
    if q_out is not None:
        desc.q_out, desc.q_out_stride_token, desc.q_out_stride_head = _ptr(q_out), hq * d, d
        desc.k_out, desc.k_out_stride_token, desc.k_out_stride_head = _ptr(k_out), k.shape[1] * d, d
    _positions_args(desc, T, dev, cu_seqlens, position_ids, seq_used)
    seg_arr, desc.n_segments = _segments_arg(segments, T)
    if seg_arr is not None:
        desc.segments = seg_arr
    desc.n_q_heads, desc.n_kv_heads, desc.head_dim = hq, k.shape[1], d
    desc.total_tokens, desc.token_offset = T, int(token_offset)
    desc.theta, desc.position_scale = float(theta), float(position_scale)
    if cache is not None:
        desc.cos_sin_cache = cache
    desc.backward = 1 if backward else 0
    if workspace is None:
        # no workspace: the library's own static staging array (rope_qk_host_static)
        st = _on(dev, load_library().rope_qk_host_static, ctypes.byref(desc), _stream(stream, dev))
        _check("rope_qk_host_static", st)
    else:
        nbytes = workspace.numel() * workspace.element_size()
        st = _on(dev, load_library().rope_qk_host, ctypes.byref(desc), _ptr(workspace), nbytes,
                 _stream(stream, dev))
        _check("rope_qk_host", st)
    return (q, k) if q_out is None else (q_out, k_out)
