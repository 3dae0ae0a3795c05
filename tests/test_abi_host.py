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
                   'int main(void) { return ROPE_QK_ABI_VERSION == 4 && GLU_GEGLU_TANH == 2 && ROPE_FLAG_POSITION_IDS_INT64 == 1 ? 0 : 1; }\n')
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.dirname(HEADER),
                           "-c", str(src), "-o", str(tmp_path / "use_header.o")])


def test_abi_version_and_strerror(lib):
    assert lib.rope_qk_abi_version() == 4
    for code in (OK, ERR_NULL, ERR_SHAPE, ERR_HEAD_DIM, ERR_ALIGN, ERR_OVERLAP, ERR_UNSUPPORTED,
                 ERR_LAUNCH, ERR_THETA, -9, -10):
        assert lib.rope_strerror(code)
    assert lib.rope_strerror(-99) == b"unknown rope status"


def test_inv_freq_matches_oracle_bits(lib, oracle_mod):
    from packed_varlen_rope_gb300 import rope_qk_inv_freq

    for theta in (1.0e4, 5.0e5, 1.0e6, 2.0, 123456.789, 1.0e9):
        for d in range(16, 257, 16):
            for scale in (1.0, 4.0, 2.5, 0.5, 7.0):
                assert np.array_equal(rope_qk_inv_freq(theta, d, scale),
                                      oracle_mod.inv_freq(theta, d, scale)), (theta, d, scale)


def test_desc_layout_matches_header(tmp_path):
    """The ctypes mirror of rope_qk_desc has the C struct's offsets and size."""
    from packed_varlen_rope_gb300 import RopeQKDesc

    names = [f[0] for f in RopeQKDesc._fields_]
    body = "".join('printf("%%zu\\n", offsetof(rope_qk_desc, %s));' % n for n in names)
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "rope_qk.h"\n'
                   'int main(void) { %s printf("%%zu\\n", sizeof(rope_qk_desc)); return 0; }\n' % body)
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c99", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)])
    got = [int(v) for v in subprocess.check_output([str(exe)]).split()]
    want = [getattr(RopeQKDesc, n).offset for n in names] + [ctypes.sizeof(RopeQKDesc)]
    assert got == want


def test_cache_bytes(lib):
    assert lib.rope_cos_sin_cache_bytes(4096, 128) == 4096 * 128 * 4
    assert lib.rope_cos_sin_cache_bytes(-1, 128) == -1
    assert lib.rope_cos_sin_cache_bytes(10, 72) == -1


# fake, never-dereferenced device addresses
Q, K, QO, KO, CU, CACHE = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000, 0x60000000


def call(lib, fn="rope_qk_fwd", q=Q, k=K, cu=CU, n=4, T=0, hq=4, hkv=2, d=64, theta=1e4, in_place=1,
         qo=None, ko=None, cache=None, rows=0):
    return getattr(lib, fn)(q, k, cu, n, T, hq, hkv, d, theta, in_place, qo, ko, cache, rows, None)


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
    assert c(rows=-5) == ERR_SHAPE
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
    assert c(cache=CACHE + 4, rows=16) == ERR_ALIGN
    assert c(cache=CACHE + 8, rows=16) == ERR_ALIGN
    assert c(T=0, in_place=0, qo=QO, ko=KO) == OK
    T = 16
    qbytes = T * 4 * 64 * 2
    assert c(T=T, k=Q + qbytes - 16) == ERR_OVERLAP
    assert c(T=T, in_place=0, qo=Q, ko=KO) == ERR_OVERLAP
    assert c(T=T, in_place=0, qo=QO, ko=QO + 16) == ERR_OVERLAP
    assert c(T=T, in_place=0, qo=QO, ko=K + 32) == ERR_OVERLAP


def test_other_entry_points_argument_checks(lib):
    assert lib.rope_cos_sin_cache_build(CACHE, 0, 128, 1e6, None) == OK
    assert lib.rope_cos_sin_cache_build(CACHE, -1, 128, 1e6, None) == ERR_SHAPE
    assert lib.rope_cos_sin_cache_build(CACHE, 8, 100, 1e6, None) == ERR_HEAD_DIM
    assert lib.rope_cos_sin_cache_build(CACHE, 8, 128, 0.0, None) == ERR_THETA
    assert lib.rope_cos_sin_cache_build(CACHE, (1 << 24) + 1, 128, 1e6, None) == ERR_UNSUPPORTED
    assert lib.rope_cos_sin_cache_build(None, 8, 128, 1e6, None) == ERR_NULL
    assert lib.rope_cos_sin_cache_build(CACHE + 8, 8, 128, 1e6, None) == ERR_ALIGN
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
    assert lib.rope_cos_sin_cache_build_scaled(CACHE, 8, 128, 1e6, -2.0, None) == ERR_THETA
    assert lib.rope_cos_sin_cache_build_scaled(CACHE, 0, 128, 1e6, 4.0, None) == OK


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
