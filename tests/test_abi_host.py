"""The C ABI without a GPU: exports, header validity, host-side argument checks.

Every call here returns before the library touches the CUDA runtime (rejected
arguments, or an empty pack), so it runs on a machine with no GPU.
"""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rope_qk.h")
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))

OK, ERR_NULL, ERR_SHAPE, ERR_HEAD_DIM, ERR_ALIGN, ERR_OVERLAP, ERR_UNSUPPORTED, ERR_LAUNCH, ERR_THETA = \
    0, -1, -2, -3, -4, -5, -6, -7, -8
ERR_WORKSPACE, ERR_CACHE = -10, -11


@pytest.fixture(scope="module")
def lib():
    from packed_varlen_rope_gb300 import build, load_library

    build.build()
    return load_library()


def declared_functions():
    names = []
    for path in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?(?:int|int64_t|char|void)\s*\*?\s*((?:rope|glu)_\w+)\s*\(",
                            text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_binding_exports():
    from packed_varlen_rope_gb300 import EXPORTS

    assert sorted(EXPORTS) == declared_functions()


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True).stdout
    for n in declared_functions():
        assert re.search(r"\bT %s$" % n, out, flags=re.M), n


def test_header_is_plain_c(tmp_path):
    src = tmp_path / "use_header.c"
    src.write_text('#include "rope_qk.h"\n#include "glu.h"\n'
                   'int main(void) { return ROPE_QK_ABI_VERSION == 5 && GLU_GEGLU_TANH == 2 && ROPE_FLAG_POSITION_IDS_INT64 == 1 &&\n'
                   '    ROPE_MAX_SEGMENTS == 16 && ROPE_ERR_CACHE == -11 ? 0 : 1; }\n')
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.dirname(HEADER),
                           "-c", str(src), "-o", str(tmp_path / "use_header.o")])


def test_abi_version_and_strerror(lib):
    assert lib.rope_qk_abi_version() == 5
    for code in (OK, ERR_NULL, ERR_SHAPE, ERR_HEAD_DIM, ERR_ALIGN, ERR_OVERLAP, ERR_UNSUPPORTED,
                 ERR_LAUNCH, ERR_THETA, -9, ERR_WORKSPACE, ERR_CACHE):
        assert lib.rope_strerror(code)
    assert lib.rope_strerror(-99) == b"unknown rope status"


def test_inv_freq_matches_oracle_bits(lib, oracle_mod):
    from packed_varlen_rope_gb300 import rope_qk_inv_freq

    for theta in (1.0e4, 5.0e5, 1.0e6, 2.0, 123456.789, 1.0e9):
        for d in range(16, 257, 16):
            for scale in (1.0, 4.0, 2.5, 0.5, 7.0):
                assert np.array_equal(rope_qk_inv_freq(theta, d, scale),
                                      oracle_mod.inv_freq(theta, d, scale)), (theta, d, scale)


@pytest.mark.parametrize("struct", ["rope_qk_desc", "rope_cos_sin_cache", "rope_qk_segment"])
def test_desc_layout_matches_header(tmp_path, struct):
    """The ctypes mirrors of the C structs have the C compiler's offsets and sizes."""
    from packed_varlen_rope_gb300 import RopeCosSinCacheDesc, RopeQKDesc, RopeQKSegment

    cls = {"rope_qk_desc": RopeQKDesc, "rope_cos_sin_cache": RopeCosSinCacheDesc,
           "rope_qk_segment": RopeQKSegment}[struct]
    names = [f[0] for f in cls._fields_]
    body = "".join('printf("%%zu\\n", offsetof(%s, %s));' % (struct, n) for n in names)
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "rope_qk.h"\n'
                   'int main(void) { %s printf("%%zu\\n", sizeof(%s)); return 0; }\n' % (body, struct))
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c99", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)])
    got = [int(v) for v in subprocess.check_output([str(exe)]).split()]
    want = [getattr(cls, n).offset for n in names] + [ctypes.sizeof(cls)]
    assert got == want


def test_cache_bytes(lib):
    assert lib.rope_cos_sin_cache_bytes(4096, 128) == 4096 * 128 * 4
    assert lib.rope_cos_sin_cache_bytes(-1, 128) == -1
    assert lib.rope_cos_sin_cache_bytes(10, 72) == -1


# fake, never-dereferenced device addresses
Q, K, QO, KO, CU, CACHE = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000, 0x60000000


def cache_desc(lib, rows=0, d=64, theta=1e4, scale=1.0, data=None):
    """A cache descriptor written by the library's build.  rows == 0 makes no CUDA call
    (no table to fill); rows > 0 is forged from a 0-row build and resealed by the
    test's own copy of the check word, to exercise the host checks without a GPU."""
    from packed_varlen_rope_gb300 import RopeCosSinCacheDesc

    c = RopeCosSinCacheDesc()
    assert lib.rope_cos_sin_cache_build(ctypes.byref(c), data, 0, d, theta, scale, None) == OK
    if rows:
        c.rows, c.data, c.device = rows, data, 0
        c.check = _fnv_check(c)
    return c


def _fnv_check(c):
    import struct

    h = 1469598103934665603
    raw = struct.pack("<Qqiidd", c.data or 0, c.rows, c.head_dim, c.device, c.theta, c.position_scale)
    for b in raw:
        h = ((h ^ b) * 1099511628211) & 0xFFFFFFFFFFFFFFFF
    return h


def call(lib, fn="rope_qk_fwd", q=Q, k=K, cu=CU, n=4, T=0, hq=4, hkv=2, d=64, theta=1e4, in_place=1,
         qo=None, ko=None, cache=None):
    return getattr(lib, fn)(q, k, cu, n, T, hq, hkv, d, theta, in_place, qo, ko,
                            None if cache is None else ctypes.pointer(cache), None)


@pytest.mark.parametrize("fn", ["rope_qk_fwd", "rope_qk_bwd"])
def test_argument_checks(lib, fn):
    # every call below is rejected on the host, before anything could be launched
    c = lambda **kw: call(lib, fn=fn, **{"T": 16, **kw})  # noqa: E731
    assert c(T=0) == OK                                  # empty pack: nothing launched
    assert c(T=0, q=None, k=None, cu=None) == OK         # ... and no pointer is read
    assert c(T=-1) == ERR_SHAPE
    assert c(n=-1) == ERR_SHAPE
    assert c(hq=0) == ERR_SHAPE
    assert c(hkv=0) == ERR_SHAPE
    for d in (0, 8, 24, 65, 72, 272, 512):
        assert c(d=d) == ERR_HEAD_DIM, d
    for th in (0.0, -1.0, float("nan"), float("inf")):
        assert c(theta=th) == ERR_THETA
    assert c(T=(1 << 24) + 1) == ERR_UNSUPPORTED
    assert c(q=None) == ERR_NULL
    assert c(k=None) == ERR_NULL
    assert c(cu=None) == ERR_NULL
    assert c(in_place=0) == ERR_NULL
    assert c(in_place=0, qo=QO) == ERR_NULL
    assert c(q=Q + 8) == ERR_ALIGN
    assert c(k=K + 2) == ERR_ALIGN
    assert c(in_place=0, qo=QO + 4, ko=KO) == ERR_ALIGN
    assert c(cache=cache_desc(lib, rows=16, data=CACHE + 4)) == ERR_ALIGN
    assert c(cache=cache_desc(lib, rows=16, data=CACHE + 8)) == ERR_ALIGN
    assert c(T=0, in_place=0, qo=QO, ko=KO) == OK
    T = 16
    qbytes = T * 4 * 64 * 2
    assert c(T=T, k=Q + qbytes - 16) == ERR_OVERLAP
    assert c(T=T, in_place=0, qo=Q, ko=KO) == ERR_OVERLAP
    assert c(T=T, in_place=0, qo=QO, ko=QO + 16) == ERR_OVERLAP
    assert c(T=T, in_place=0, qo=QO, ko=K + 32) == ERR_OVERLAP


def test_other_entry_points_argument_checks(lib):
    from packed_varlen_rope_gb300 import RopeCosSinCacheDesc

    c = RopeCosSinCacheDesc()
    b = lambda data=CACHE, rows=8, d=128, theta=1e6, scale=1.0, out=ctypes.byref(c): \
        lib.rope_cos_sin_cache_build(out, data, rows, d, theta, scale, None)  # noqa: E731
    assert b(rows=0) == OK
    assert b(rows=-1) == ERR_SHAPE
    assert b(d=100) == ERR_HEAD_DIM
    assert b(theta=0.0) == ERR_THETA
    assert b(scale=-2.0) == ERR_THETA and b(scale=float("inf")) == ERR_THETA
    assert b(rows=(1 << 24) + 1) == ERR_UNSUPPORTED
    assert b(data=None) == ERR_NULL
    assert b(data=CACHE + 8) == ERR_ALIGN
    assert b(out=None) == ERR_NULL
    assert b(rows=0, scale=4.0) == OK
    assert lib.rope_qk_positions(CU, 3, 0, Q, None) == OK
    assert lib.rope_qk_positions(CU, -1, 8, Q, None) == ERR_SHAPE
    assert lib.rope_qk_positions(None, 3, 8, Q, None) == ERR_NULL
    assert lib.rope_qk_positions(CU, 3, 8, None, None) == ERR_NULL
    assert lib.rope_qk_positions(CU, 3, (1 << 24) + 1, Q, None) == ERR_UNSUPPORTED
    assert lib.rope_validate_cu_seqlens(None, 3, 8, Q, None) == ERR_NULL
    assert lib.rope_validate_cu_seqlens(CU, 3, 8, None, None) == ERR_NULL
    assert lib.rope_validate_cu_seqlens(CU, -2, 8, Q, None) == ERR_SHAPE
    w = (ctypes.c_float * 64)()
    assert lib.rope_qk_inv_freq(1e4, 100, 1.0, w) == ERR_HEAD_DIM
    assert lib.rope_qk_inv_freq(1e4, 128, 1.0, None) == ERR_NULL
    assert lib.rope_qk_inv_freq(1e4, 128, 0.0, w) == ERR_THETA


def test_cache_descriptor_must_match_the_call(lib):
    """A cache serves only the (theta, head_dim, position_scale) it was built for, and
    only as the build wrote it: every mismatch is ROPE_ERR_CACHE, found on the host."""
    from packed_varlen_rope_gb300 import RopeCosSinCacheDesc

    c = RopeCosSinCacheDesc()
    assert lib.rope_cos_sin_cache_build(ctypes.byref(c), None, 0, 64, 1e4, 1.0, None) == OK
    assert (c.rows, c.head_dim, c.theta, c.position_scale, c.device) == (0, 64, 1e4, 1.0, -1)
    assert c.check == _fnv_check(c)          # the test's copy of the check word agrees
    f = lambda cache, **kw: call(lib, T=16, cache=cache, **kw)  # noqa: E731
    assert f(cache_desc(lib, rows=0)) != ERR_CACHE      # matching (and empty): accepted by the checks
    assert f(cache_desc(lib, theta=1e6)) == ERR_CACHE
    assert f(cache_desc(lib, d=128)) == ERR_CACHE
    assert f(cache_desc(lib, scale=4.0)) == ERR_CACHE               # the plain entry points use scale 1
    forged = cache_desc(lib)
    forged.rows = 1 << 20                                           # changed after the build
    assert f(forged) == ERR_CACHE
    forged = cache_desc(lib)
    forged.theta = 1e6                                              # ... to match another call
    assert call(lib, T=16, theta=1e6, cache=forged) == ERR_CACHE
    assert f(RopeCosSinCacheDesc()) == ERR_CACHE                    # never built (all zero)
    # the descriptor form checks position_scale against the cache as well
    a = lambda **kw: lib.rope_qk_apply(ctypes.byref(_desc(**kw)), None)  # noqa: E731
    scaled = cache_desc(lib, scale=4.0)
    assert a(position_scale=4.0, cos_sin_cache=ctypes.pointer(scaled)) != ERR_CACHE
    assert a(position_scale=2.0, cos_sin_cache=ctypes.pointer(scaled)) == ERR_CACHE
    assert a(position_scale=4.0, theta=1e5, cos_sin_cache=ctypes.pointer(scaled)) == ERR_CACHE
    # host-buffer entries reject it before any copy
    for entry in ("rope_qk_host", "rope_qk_host_static"):
        d = _desc(cos_sin_cache=ctypes.pointer(cache_desc(lib, theta=7.0)))
        args = (ctypes.byref(d),) + ((Q, 1 << 20) if entry == "rope_qk_host" else ()) + (None,)
        assert getattr(lib, entry)(*args) == ERR_CACHE


def _desc(T=16, hq=4, hkv=2, d=64, **kw):
    from packed_varlen_rope_gb300 import RopeQKDesc

    p = RopeQKDesc()
    p.q, p.q_stride_token, p.q_stride_head = Q, hq * d, d
    p.k, p.k_stride_token, p.k_stride_head = K, hkv * d, d
    p.cu_seqlens, p.n_seqs = CU, 3
    p.n_q_heads, p.n_kv_heads, p.head_dim = hq, hkv, d
    p.total_tokens, p.theta, p.position_scale = T, 1e4, 1.0
    for key, v in kw.items():
        setattr(p, key, v)
    return p


def test_apply_argument_checks(lib):
    """rope_qk_apply rejections (every one happens on the host, before any launch)."""
    a = lambda **kw: lib.rope_qk_apply(ctypes.byref(_desc(**kw)), None)  # noqa: E731
    assert lib.rope_qk_apply(None, None) == ERR_NULL
    assert a(T=0) == OK
    assert a(T=0, q=None, k=None, cu_seqlens=None) == OK
    assert a(position_scale=0.0) == ERR_THETA
    assert a(position_scale=float("nan")) == ERR_THETA
    assert a(token_offset=-1) == ERR_SHAPE
    assert a(token_offset=(1 << 24) - 8) == ERR_UNSUPPORTED        # global tokens past 2^24
    assert a(cu_seqlens=None) == ERR_NULL
    assert a(flags=2) == ERR_UNSUPPORTED and a(T=0, flags=4) == ERR_UNSUPPORTED   # unknown flag bits
    assert a(flags=1, position_ids=CU + 4) == ERR_ALIGN              # int64 ids need 8-byte alignment
    for entry in ("rope_qk_host", "rope_qk_host_static"):            # the host entries check them too
        args = (ctypes.byref(_desc(flags=2)),) + ((Q, 1 << 20) if entry == "rope_qk_host" else ()) + (None,)
        assert getattr(lib, entry)(*args) == ERR_UNSUPPORTED
    assert a(q_stride_token=4 * 64 + 4) == ERR_ALIGN                # stride not a multiple of 8
    assert a(k_stride_head=60) == ERR_ALIGN
    assert a(q_stride_head=56) == ERR_OVERLAP                       # heads overlap (stride < d)
    assert a(q_stride_token=128) == ERR_OVERLAP                     # tokens overlap the 4 heads
    assert a(q_stride_token=-256) == ERR_SHAPE
    assert a(q_stride_token=1 << 60) == ERR_SHAPE                   # span would overflow int64 bytes
    assert a(k_stride_head=1 << 58, hkv=2) == ERR_SHAPE
    # fused QKV buffer: Q and K slices may interleave, but not share elements
    S = (4 + 2 * 2) * 64
    assert a(q_stride_token=S, k=Q + 3 * 64 * 2, k_stride_token=S) == ERR_OVERLAP   # K starts inside Q
    assert a(q_stride_token=S, k=Q + 4 * 64 * 2, k_stride_token=S + 8) == ERR_OVERLAP  # strides differ
    # out of place: both outputs or none, and outputs away from inputs
    assert a(q_out=QO) == ERR_NULL
    assert a(q_out=QO, q_out_stride_token=256, q_out_stride_head=64, k_out=Q, k_out_stride_token=128,
             k_out_stride_head=64) == ERR_OVERLAP


def test_glu_argument_checks(lib):
    ERR_KIND = -9
    E, G, H, DH = 0x10000000, 0x20000000, 0x30000000, 0x40000000
    f = lambda kind=0, e=E, es=64, g=G, gs=64, h=H, hs=64, rows=4, cols=64: \
        lib.glu_fwd(kind, e, es, g, gs, h, hs, rows, cols, None)  # noqa: E731
    assert f(rows=0) == OK and f(cols=0) == OK
    assert f(kind=3) == ERR_KIND and f(kind=-1) == ERR_KIND
    assert f(rows=-1) == ERR_SHAPE and f(cols=12) == ERR_SHAPE and f(es=32) == ERR_SHAPE
    assert f(rows=1 << 20, cols=1 << 14) == ERR_SHAPE                      # units >= 2^31
    assert f(es=64 + (1 << 31)) == ERR_SHAPE                               # stride - cols >= 2^31
    assert f(es=64 + (1 << 31), rows=1) != ERR_SHAPE                       # one row: stride unused
    assert f(rows=1 << 28, cols=8, es=1 << 31, gs=8, hs=8) == ERR_SHAPE     # span 2^59 elements
    assert f(e=None) == ERR_NULL and f(h=None) == ERR_NULL
    assert f(e=E + 8) == ERR_ALIGN and f(gs=68) == ERR_ALIGN
    assert f(h=E + 64) == ERR_OVERLAP                                      # partial overlap
    assert f(h=E, hs=128) == ERR_OVERLAP                                   # same start, other stride
    b = lambda de=E + 0x8000000, dg=G + 0x8000000, **kw: lib.glu_bwd(  # noqa: E731
        kw.get("kind", 0), DH, 64, E, 64, G, 64, de, 64, dg, 64, 4, 64, None)
    assert b(de=H, dg=H) == ERR_OVERLAP                                    # outputs collide
    # side-by-side halves of one [4, 128] buffer are disjoint; shifted by 8 they are not
    fused = lambda off: lib.glu_fwd(0, E, 128, E + 128, 128, E + off, 128, 4, 64, None)  # noqa: E731
    assert fused(16) == ERR_OVERLAP and fused(64) == ERR_OVERLAP
    assert b(de=DH + 16) == ERR_OVERLAP
    assert b(kind=7) == ERR_KIND


def test_binding_rejects_cpu_tensors():
    import torch

    import packed_varlen_rope_gb300 as pr

    q = torch.zeros(4, 2, 64, dtype=torch.bfloat16)
    k = torch.zeros(4, 1, 64, dtype=torch.bfloat16)
    cu = torch.tensor([0, 4], dtype=torch.int32)
    with pytest.raises(ValueError):
        pr.rope_qk_fwd(q, k, cu, 1e4)


def test_rotary_cache_growth_rule():
    from packed_varlen_rope_gb300 import cache_rows_for

    assert cache_rows_for(1, 0) == 1024 and cache_rows_for(1024, 0) == 1024
    assert cache_rows_for(1025, 1024) == 2048 and cache_rows_for(16384, 0) == 16384
    assert cache_rows_for(20000, 16384) == 32768 and cache_rows_for(500, 32768) == 32768
    assert cache_rows_for((1 << 20) + 1, 1 << 20) == 1 << 21


def test_segment_list_checks(lib):
    """rope_qk_apply's segment list: starts at row 0, rows strictly increasing and inside
    the call, tokens non-negative and below 2^24; it needs cu_seqlens and offset 0."""
    from packed_varlen_rope_gb300 import RopeQKSegment

    def a(segs, **kw):
        arr = (RopeQKSegment * max(1, len(segs)))(*[RopeQKSegment(r, t) for r, t in segs])
        p = _desc(**kw)
        p.segments, p.n_segments = arr, len(segs)
        return lib.rope_qk_apply(ctypes.byref(p), None)

    assert a([(1, 0)]) == ERR_SHAPE                        # does not start at row 0
    assert a([(0, 0), (8, 100), (8, 200)]) == ERR_SHAPE    # row_start not increasing
    assert a([(0, 0), (16, 100)]) == ERR_SHAPE             # a segment starting past the rows
    assert a([(0, -1)]) == ERR_SHAPE
    assert a([(0, 0), (8, (1 << 24) - 4)]) == ERR_UNSUPPORTED   # last token of segment 2 past 2^24
    assert a([(0, 0)], token_offset=4) == ERR_SHAPE
    assert a([(0, 0)], position_ids=CU) == ERR_UNSUPPORTED
    p = _desc()
    p.n_segments = 17
    assert lib.rope_qk_apply(ctypes.byref(p), None) == ERR_SHAPE
    p.n_segments = 2                                       # segments pointer left NULL
    assert lib.rope_qk_apply(ctypes.byref(p), None) == ERR_NULL
    p.n_segments, p.reserved = 0, 1
    assert lib.rope_qk_apply(ctypes.byref(p), None) == ERR_UNSUPPORTED


@pytest.mark.parametrize("entry", ["rope_qk_host", "rope_qk_host_static"])
def test_host_entries_check_the_whole_pack_first(lib, entry):
    """A host-buffer call whose pack crosses 2^24 global tokens only in a late chunk is
    rejected before any copy: the status is the argument error (a CUDA call on this
    machine, which has no GPU, would have failed with ROPE_ERR_LAUNCH), and the host
    buffers are untouched."""
    from packed_varlen_rope_gb300 import RopeQKDesc, RopeQKSegment

    T, hq, hkv, d = 4096, 2, 1, 64
    q = np.arange(T * hq * d, dtype=np.uint16).reshape(T, hq, d)
    k = np.arange(T * hkv * d, dtype=np.uint16).reshape(T, hkv, d) ^ 0x5555
    q0, k0 = q.copy(), k.copy()
    p = RopeQKDesc()
    p.q, p.q_stride_token, p.q_stride_head = q.ctypes.data, hq * d, d
    p.k, p.k_stride_token, p.k_stride_head = k.ctypes.data, hkv * d, d
    p.cu_seqlens, p.n_seqs = CU, 1
    p.n_q_heads, p.n_kv_heads, p.head_dim = hq, hkv, d
    p.total_tokens, p.theta, p.position_scale = T, 1e4, 1.0
    extra = (Q, 64 * 1024) if entry == "rope_qk_host" else ()      # a workspace of many chunks
    run = lambda: getattr(lib, entry)(ctypes.byref(p), *extra, None)  # noqa: E731
    p.token_offset = (1 << 24) - T + 1                              # only the last token is past 2^24
    assert run() == ERR_UNSUPPORTED
    p.token_offset = 0
    segs = (RopeQKSegment * 2)(RopeQKSegment(0, 0), RopeQKSegment(T - 8, (1 << 24) - 4))
    p.segments, p.n_segments = segs, 2                              # the second segment crosses it
    assert run() == ERR_UNSUPPORTED
    p.segments, p.n_segments = None, 0
    p.theta = -1.0
    assert run() == ERR_THETA
    p.theta, p.q_stride_head = 1e4, d + 8                           # host buffers must be contiguous
    assert run() == ERR_SHAPE
    assert np.array_equal(q, q0) and np.array_equal(k, k0)


def test_host_binding_checks_outputs_and_cache():
    """rope_qk_host rejects output buffers of another shape and a cache of the wrong
    type, dtype, shape or device with ValueError before any C call."""
    import torch

    import packed_varlen_rope_gb300 as pr
    from packed_varlen_rope_gb300 import CosSinCache, RopeCosSinCacheDesc

    T, hq, hkv, d = 32, 4, 2, 64
    q = torch.zeros(T, hq, d, dtype=torch.bfloat16)
    k = torch.zeros(T, hkv, d, dtype=torch.bfloat16)
    cu = torch.tensor([0, T], dtype=torch.int32)
    for qo, ko in ((torch.zeros(T - 1, hq, d, dtype=torch.bfloat16), torch.zeros(T, hkv, d, dtype=torch.bfloat16)),
                   (torch.zeros(T, hq, d, dtype=torch.bfloat16), torch.zeros(T, hkv, d // 2, dtype=torch.bfloat16)),
                   (torch.zeros(T, hq, d, dtype=torch.bfloat16), torch.zeros(T, hkv + 1, d, dtype=torch.bfloat16))):
        with pytest.raises(ValueError, match="shapes"):
            pr.rope_qk_host(q, k, 1e4, cu_seqlens=cu, q_out=qo, k_out=ko, device="cuda:0")

    def cache(t, rows=None):
        desc = RopeCosSinCacheDesc()
        desc.rows = t.shape[0] if rows is None else rows
        return CosSinCache(t, desc)

    bad = [
        (torch.zeros(8, 4, d // 16, 4, dtype=torch.float32), "cos_sin_cache must be a CosSinCache"),
        (cache(torch.zeros(8, 4, d // 16, 4, dtype=torch.bfloat16)), "float32"),
        (cache(torch.zeros(8, 4, d // 16, 4, dtype=torch.float16)), "float32"),
        (cache(torch.zeros(8, 4, d // 32, 4, dtype=torch.float32)), "head_dim 64"),       # built for d = 32
        (cache(torch.zeros(8, 4, d // 16, 4, dtype=torch.float32), rows=16), "rows"),     # table shorter than claimed
        (cache(torch.zeros(8, 4, 2 * d // 16, 4, dtype=torch.float32)[:, :, ::2]), "contiguous"),
        (cache(torch.zeros(8, 4, d // 16, 4, dtype=torch.float32)), "is on cpu"),          # host memory
    ]
    for c, why in bad:
        with pytest.raises(ValueError, match=why if why != "rows" else "table"):
            pr.rope_qk_host(q, k, 1e4, cu_seqlens=cu, cos_sin_cache=c, device="cuda:0")


def test_cp_shard_plan():
    """Contiguous and load-balanced context-parallel shards cover every token of the
    padded pack exactly once; rank r of the load-balanced plan holds chunks r and
    2 cp - 1 - r; the segments map local rows to those tokens."""
    from packed_varlen_rope_gb300 import cp_shards, shard_rows, shard_segments

    for T in (0, 1, 7, 64, 1000, 65536, 65537):
        for cp in (1, 2, 3, 4, 8):
            for lb in (False, True):
                rows = [shard_rows(cp_shards(T, cp, r, lb)) for r in range(cp)]
                flat = sorted(t for rr in rows for t in rr)
                n_chunks = 2 * cp if lb else cp
                padded = -(-T // n_chunks) * n_chunks
                assert flat == list(range(padded)), (T, cp, lb)
                assert len({len(rr) for rr in rows}) == 1          # equal shards (padding included)
                for r in range(cp):
                    sh = cp_shards(T, cp, r, lb)
                    segs = shard_segments(sh)
                    local = shard_rows(sh)
                    for i, (row0, tok0) in enumerate(segs):
                        row1 = segs[i + 1][0] if i + 1 < len(segs) else len(local)
                        assert local[row0:row1] == list(range(tok0, tok0 + row1 - row0))
    c = -(-1000 // 8)
    assert cp_shards(1000, 4, 1) == [(c, c), (6 * c, c)]
    assert shard_segments(cp_shards(1000, 4, 1)) == [(0, c), (c, 6 * c)]
    with pytest.raises(ValueError):
        cp_shards(10, 2, 2)


def test_launch_info_names_the_dispatched_instance(lib):
    """rope_qk_launch_info reports the kernel instance rope_qk_apply picks: the head_dim
    template (64, 96, 128, 256, else the generic 0) and 64-bit offsets exactly when a
    view spans 2^31 elements or more -- the 1M-token pack (32 Q heads of 128) needs
    them, the 65,536-token Qwen3-32B pack does not."""
    from packed_varlen_rope_gb300 import RopeQKDesc, RopeQKLaunch

    def info(T, hq, hkv, d, **kw):
        p = RopeQKDesc()
        p.q, p.q_stride_token, p.q_stride_head = 1 << 40, hq * d, d
        p.k, p.k_stride_token, p.k_stride_head = 1 << 44, hkv * d, d
        p.cu_seqlens, p.n_seqs = CU, 1
        p.n_q_heads, p.n_kv_heads, p.head_dim = hq, hkv, d
        p.total_tokens, p.theta, p.position_scale = T, 1e6, 1.0
        for key, v in kw.items():
            setattr(p, key, v)
        out = RopeQKLaunch()
        assert lib.rope_qk_launch_info(ctypes.byref(p), ctypes.byref(out)) == OK
        return out

    w4 = info(65536, 64, 8, 128)
    assert w4.kernel_name() == "rope_qk_tile_kernel<128,false,2>"          # no cache: 2 units per thread
    assert (w4.tile_tokens, w4.threads, w4.grid, w4.unroll) == (1, 128, 65536, 2)
    # with a cos/sin cache, a launch of at least 32,768 tiles keeps 4 units per thread in flight
    cache = cache_desc(lib, rows=4096, d=128, theta=1e6, data=CACHE)
    assert info(65536, 64, 8, 128, cos_sin_cache=ctypes.pointer(cache)).kernel_name() == \
        "rope_qk_tile_kernel<128,false,4>"
    assert info(32768, 64, 8, 128, cos_sin_cache=ctypes.pointer(cache)).unroll == 4   # exactly 32,768 tiles
    assert info(32767, 64, 8, 128, cos_sin_cache=ctypes.pointer(cache)).unroll == 2
    w2 = info(16384, 32, 8, 128, cos_sin_cache=ctypes.pointer(cache))
    assert (w2.unroll, w2.tile_tokens, w2.grid) == (3, 1, 16384)        # 320 units a token, 256 a tile
    assert w2.kernel_name() == "rope_qk_tile_kernel<128,false,3>"       # the tile in one batch of 3
    # ... as long as the launch stays below 32,768 such tiles; a larger one keeps 512 a tile
    assert info(32767, 32, 8, 128, cos_sin_cache=ctypes.pointer(cache)).tile_tokens == 1
    big = info(32768, 32, 8, 128, cos_sin_cache=ctypes.pointer(cache))
    assert (big.tile_tokens, big.grid, big.unroll) == (2, 16384, 2)
    # without a cache a tile holds about 512 units (2 tokens of 320), under seq_used 1,024
    assert info(16384, 32, 8, 128).tile_tokens == 2
    su = info(16384, 32, 8, 128, cos_sin_cache=ctypes.pointer(cache), seq_used=1 << 46)
    assert (su.tile_tokens, su.unroll, su.grid) == (4, 2, 4096)                # seq_used: about 1,024 units
    assert info(16384, 32, 8, 128).unroll == 2                                  # no cache
    assert info(16384, 4, 2, 64, cos_sin_cache=ctypes.pointer(cache_desc(lib, rows=64, d=64, theta=1e6,
                                                                          data=CACHE))).tile_tokens == 11
    w5 = info(1 << 20, 32, 8, 128)
    assert w5.kernel_name() == "rope_qk_tile_kernel<128,true,2>" and w5.grid == (1 << 20) // w5.tile_tokens
    assert info(1 << 20, 32, 8, 128, cos_sin_cache=ctypes.pointer(cache)).kernel_name() == \
        "rope_qk_tile_kernel<128,true,3>"                                  # 64-bit offsets, a cache: 3
    assert info(4096, 4, 2, 80).kernel_name() == "rope_qk_tile_kernel<0,false,2>"
    assert info(1 << 16, 64, 8, 80, cos_sin_cache=ctypes.pointer(cache_desc(lib, rows=64, d=80, theta=1e6,
                                                                              data=CACHE))).unroll == 2  # generic
    assert info(64, 4, 2, 64).kernel_name() == "rope_qk_tile_kernel<64,false,2>"
    # head-major views of 2^19 tokens x 32 heads: the head stride makes the span pass 2^31
    hm = info(1 << 19, 32, 8, 128, q_stride_token=128, q_stride_head=(1 << 19) * 128)
    assert hm.long_index == 1
    empty = info(0, 4, 2, 64)
    assert empty.grid == 0
    assert lib.rope_qk_launch_info(None, ctypes.byref(RopeQKLaunch())) == ERR_NULL
    p = RopeQKDesc()
    assert lib.rope_qk_launch_info(ctypes.byref(p), None) == ERR_NULL


def test_cos_sin_eval_argument_checks(lib):
    e = lambda phi=Q, c=K, s=QO, n=16, mode=0: lib.rope_cos_sin_eval(phi, c, s, n, mode, None)  # noqa: E731
    assert e(n=0) == OK and e(n=0, phi=None) == OK
    assert e(n=-1) == ERR_SHAPE
    assert e(mode=3) == -9 and e(mode=-1) == -9
    assert e(phi=None) == ERR_NULL and e(c=None) == ERR_NULL and e(s=None) == ERR_NULL


def test_ulysses_head_plan():
    """Ulysses head shards: every Q head on exactly one rank; K/V heads split when there
    are enough, else each rank keeps the one its Q heads share."""
    from packed_varlen_rope_gb300 import ulysses_heads

    for hq, hkv, sp in ((64, 8, 8), (64, 8, 4), (32, 8, 16), (32, 32, 8), (64, 8, 16), (4, 2, 4)):
        seen = []
        for r in range(sp):
            (q0, q1), (k0, k1) = ulysses_heads(hq, hkv, sp, r)
            seen += list(range(q0, q1))
            group = hq // hkv
            assert all(k0 <= h // group < k1 for h in range(q0, q1)), (hq, hkv, sp, r)   # Q heads' K/V head held
        assert sorted(seen) == list(range(hq))
    assert ulysses_heads(64, 8, 16, 3) == ((12, 16), (1, 2))
    assert ulysses_heads(64, 8, 4, 1) == ((16, 32), (2, 4))
    for bad in ((64, 8, 3, 0), (64, 8, 8, 8), (12, 8, 4, 0), (64, 6, 4, 0)):
        with pytest.raises(ValueError):
            ulysses_heads(*bad)
