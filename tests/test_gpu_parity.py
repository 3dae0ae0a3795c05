"""CUDA path against the CPU oracle, element by element (needs a GB300).

Every call goes through the C ABI (librope_qk.so via its ctypes binding).  Small and
medium workloads are compared in full; the 1M-token pack (64-bit offsets) is compared
on seeded sampled rows, including the tokens where Q's flat offset crosses 2^31.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from parity_util import assert_parity, compare, from_bits, merge, to_bits

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


def pr():
    import packed_varlen_rope_gb300 as m

    return m


def _normal_bits(rng, shape, scale=1.0):
    f = torch.from_numpy((rng.standard_normal(size=shape) * scale).astype(np.float32))
    return f.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _check_full(q_bits, k_bits, cu, theta, q_gpu, k_gpu, bwd, what, exact=True):
    """Oracle over every token row of q/k; q_gpu/k_gpu are the CUDA results."""
    stats = {}
    for name, x, y in (("q", q_bits, q_gpu), ("k", k_bits, k_gpu)):
        ref = oracle.rope_packed(x, cu, theta, bwd=bwd)
        s = compare(to_bits(y), ref, x)
        assert_parity(s, (what, name))
        if exact:
            assert s["bit_mismatch"] == 0, (what, name, s)
        stats = merge(stats, s)
    return stats


def _run(fn, q, k, cu_dev, theta, cache=None, **kw):
    getattr(pr(), fn)(q, k, cu_dev, theta, cos_sin_cache=cache, **kw)
    torch.cuda.synchronize()


# ------------------------------------------------------------------ positions

def _packs_for_positions():
    from packed_varlen_rope_gb300 import workloads as wl

    packs = []
    for i in (1, 2, 4, 5):
        p = wl.make_pack(wl.WORKLOADS[i])
        packs.append((p.cu_seqlens, p.total_tokens))
    p3 = wl.make_pack(wl.WORKLOADS[3], "padded")
    packs.append((p3.cu_seqlens, p3.total_tokens))
    rng = np.random.Generator(np.random.PCG64(31))
    for _ in range(20):
        n = int(rng.integers(1, 300))
        lengths = rng.integers(0, 40, size=n)
        lengths[rng.random(n) < 0.3] = 0
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
        packs.append((cu, int(cu[-1] + rng.integers(0, 50))))
    packs.append((np.array([0], dtype=np.int32), 17))               # no samples at all
    packs.append((np.array([0, 1, 2, 3, 4, 5], dtype=np.int32), 5))  # one token each
    return packs


def test_positions_bit_exact(dev):
    for cu, T in _packs_for_positions():
        got = pr().rope_qk_positions(torch.from_numpy(cu).to(dev), T).cpu().numpy()
        assert np.array_equal(got, oracle.positions(cu, T)), (cu[:8], T)


def test_positions_nonzero_start(dev):
    cu = np.array([3, 5, 9], dtype=np.int32)
    got = pr().rope_qk_positions(torch.from_numpy(cu).to(dev), 12).cpu().numpy()
    assert got.tolist() == [-1, -1, -1, 0, 1, 0, 1, 2, 3, -1, -1, -1]


def test_validate_cu_seqlens(dev):
    m = pr()
    cases = [
        ([0, 5, 22, 55, 64], 64, 0),
        ([0, 5, 5, 64], 70, 0),
        ([0, 9, 5, 64], 64, m.ROPE_CU_DECREASING),
        ([0, 5, 80], 64, m.ROPE_CU_PAST_END),
        ([2, 5, 9], 64, m.ROPE_CU_NONZERO_START),
        ([-3, 5, 9], 64, m.ROPE_CU_NEGATIVE_START | m.ROPE_CU_NONZERO_START),
        ([0], 0, 0),
    ]
    big = np.arange(0, 3001, dtype=np.int32)
    big[2500] = 1                                                     # one drop deep inside
    cases.append((big.tolist(), 3000, m.ROPE_CU_DECREASING))
    for cu, T, want in cases:
        err = m.rope_validate_cu_seqlens(torch.tensor(cu, dtype=torch.int32, device=dev), T)
        assert int(err.item()) == want, (cu[:6], T)


# ------------------------------------------------------------------ cos/sin cache

@pytest.mark.parametrize("theta,d,rows", [(1.0e4, 64, 64), (1.0e6, 128, 8192), (5.0e5, 128, 2048)])
def test_cache_matches_oracle(dev, theta, d, rows):
    cache = pr()._binding.cache_as_cos_sin(pr().new_cos_sin_cache(rows, d, theta, device=dev).data.cpu().numpy())
    mism = 0
    for p in range(rows):
        c, s = oracle.cos_sin(p, theta, d)
        mism += int(np.count_nonzero(cache[p, :, 0] != c)) + int(np.count_nonzero(cache[p, :, 1] != s))
    assert mism == 0


def test_cache_large_positions(dev):
    theta, d = 1.0e6, 128
    rows = 1 << 20
    cache = pr().new_cos_sin_cache(rows, d, theta, device=dev)
    rng = np.random.Generator(np.random.PCG64(32))
    picks = np.unique(np.concatenate([rng.integers(0, rows, 600), [rows - 1, (1 << 19), 1]]))
    got = pr()._binding.cache_as_cos_sin(cache.data[torch.from_numpy(picks).to(dev)].cpu().numpy())
    mism = 0
    for r, p in enumerate(picks):
        c, s = oracle.cos_sin(int(p), theta, d)
        mism += int(np.count_nonzero(got[r, :, 0] != c)) + int(np.count_nonzero(got[r, :, 1] != s))
    assert mism == 0


def test_cache_every_position_matches_oracle(dev):
    """All 2^20 x 64 (cos, sin) pairs of the cache the 1M-token workload uses, against
    the oracle's binary64-then-round values: identical bits everywhere.  The oracle runs
    over position ranges on every host core (its C calls release the GIL)."""
    import concurrent.futures as cf
    import ctypes
    import os

    theta, d, rows = 1.0e6, 128, 1 << 20
    got = pr()._binding.cache_as_cos_sin(pr().new_cos_sin_cache(rows, d, theta, device=dev).data.cpu().numpy())
    ref_c = np.empty((rows, d // 2), np.float32)
    ref_s = np.empty((rows, d // 2), np.float32)
    fn = oracle.get().lib.oracle_cos_sin_scaled
    fp = ctypes.POINTER(ctypes.c_float)

    def part(lo, hi):
        for p in range(lo, hi):
            fn(p, theta, d, 1.0, ref_c[p].ctypes.data_as(fp), ref_s[p].ctypes.data_as(fp))

    n = len(os.sched_getaffinity(0))
    bounds = np.linspace(0, rows, n + 1).astype(int)
    with cf.ThreadPoolExecutor(n) as ex:
        list(ex.map(lambda i: part(bounds[i], bounds[i + 1]), range(n)))
    assert np.array_equal(got[:, :, 0], ref_c) and np.array_equal(got[:, :, 1], ref_s)


# ------------------------------------------------------------------ workloads 1-4

def _workload_inputs(idx, layout="packed"):
    from packed_varlen_rope_gb300 import workloads as wl

    w = wl.WORKLOADS[idx]
    pack = wl.make_pack(w, layout)
    T = pack.total_tokens
    q = wl.normal_bf16((T, w.n_q_heads, w.head_dim), wl.seed(idx, "q"), device="cuda")
    k = wl.normal_bf16((T, w.n_kv_heads, w.head_dim), wl.seed(idx, "k"), device="cuda")
    dq = wl.normal_bf16((T, w.n_q_heads, w.head_dim), wl.seed(idx, "dq"), device="cuda")
    dk = wl.normal_bf16((T, w.n_kv_heads, w.head_dim), wl.seed(idx, "dk"), device="cuda")
    return w, pack, q, k, dq, dk


@pytest.mark.parametrize("idx,layout", [(1, "packed"), (2, "packed"), (3, "packed"), (3, "padded")])
@pytest.mark.parametrize("use_cache", [True, False])
def test_workload_fwd_bwd_full(dev, idx, layout, use_cache):
    w, pack, q, k, dq, dk = _workload_inputs(idx, layout)
    cu_dev = torch.from_numpy(pack.cu_seqlens).to(dev)
    cache = None
    if use_cache:
        cache = pr().new_cos_sin_cache(max(pack.lengths + [1]) if layout == "packed" else pack.total_tokens,
                                       w.head_dim, w.theta, device=dev)
    q0, k0, dq0, dk0 = (to_bits(t) for t in (q, k, dq, dk))
    _run("rope_qk_fwd", q, k, cu_dev, w.theta, cache)
    _check_full(q0, k0, pack.cu_seqlens, w.theta, q, k, False, (idx, layout, "fwd"))
    _run("rope_qk_bwd", dq, dk, cu_dev, w.theta, cache)
    _check_full(dq0, dk0, pack.cu_seqlens, w.theta, dq, dk, True, (idx, layout, "bwd"))


def test_padded_equals_packed_on_gpu(dev):
    from packed_varlen_rope_gb300 import workloads as wl

    w = wl.WORKLOADS[3]
    padded = wl.make_pack(w, "padded")
    packed = wl.make_pack(w, "packed")
    x = wl.normal_bf16((padded.total_tokens, w.n_q_heads, w.head_dim), 77, device="cuda")
    valid = torch.from_numpy(np.flatnonzero(padded.valid_mask)).to(dev)
    xp = x[valid].contiguous()
    kx = torch.zeros((padded.total_tokens, w.n_kv_heads, w.head_dim), dtype=torch.bfloat16, device=dev)
    kp = kx[valid].contiguous()
    _run("rope_qk_fwd", x, kx, torch.from_numpy(padded.cu_seqlens).to(dev), w.theta)
    _run("rope_qk_fwd", xp, kp, torch.from_numpy(packed.cu_seqlens).to(dev), w.theta)
    assert torch.equal(x[valid].view(torch.int16), xp.view(torch.int16))
    # the padded layout wastes what the page's padding algebra predicts
    assert padded.valid_tokens == packed.total_tokens == sum(packed.lengths)


def test_workload4_full(dev):
    """Qwen3-32B shape, 65,536 tokens, the benchmark's launch configuration (cache, in
    place); every element compared, in token chunks."""
    idx = 4
    w, pack, q, k, dq, dk = _workload_inputs(idx)
    cu_dev = torch.from_numpy(pack.cu_seqlens).to(dev)
    cache = pr().new_cos_sin_cache(max(pack.lengths), w.head_dim, w.theta, device=dev)
    inputs = [to_bits(t) for t in (q, k, dq, dk)]
    _run("rope_qk_fwd", q, k, cu_dev, w.theta, cache)
    _run("rope_qk_bwd", dq, dk, cu_dev, w.theta, cache)
    pos = oracle.positions(pack.cu_seqlens, pack.total_tokens)
    total = {}
    for x, y, bwd in ((inputs[0], q, False), (inputs[1], k, False), (inputs[2], dq, True), (inputs[3], dk, True)):
        yb = to_bits(y)
        for a in range(0, pack.total_tokens, 8192):
            b = min(pack.total_tokens, a + 8192)
            ref = oracle.rope_rows(x[a:b], pos[a:b], w.theta, bwd=bwd)
            s = compare(yb[a:b], ref, x[a:b])
            assert_parity(s, ("w4", a, bwd))
            total = merge(total, s)
    assert total["bit_mismatch"] == 0, total


# ------------------------------------------------------------------ 1M tokens, 64-bit offsets

def test_workload5_long_sampled(dev):
    """One 1,048,576-token sequence, Q numel 2^32: the 64-bit-offset kernel.  Rows are
    checked on a seeded sample plus the rows around Q's flat offset 2^31; a canary
    after the last Q element must survive."""
    from packed_varlen_rope_gb300 import workloads as wl

    w = wl.WORKLOADS[5]
    pack = wl.make_pack(w)
    T = pack.total_tokens
    guard = 4096
    q_store = torch.empty(T * w.n_q_heads * w.head_dim + guard, dtype=torch.bfloat16, device=dev)
    q = q_store[: T * w.n_q_heads * w.head_dim].view(T, w.n_q_heads, w.head_dim)
    q.copy_(wl.normal_bf16((T, w.n_q_heads, w.head_dim), wl.seed(5, "q"), device="cuda"))
    canary = torch.full((guard,), 7.25, dtype=torch.bfloat16, device=dev)
    q_store[-guard:].copy_(canary)
    k = wl.normal_bf16((T, w.n_kv_heads, w.head_dim), wl.seed(5, "k"), device="cuda")
    rows = wl.sampled_rows(w)
    rows_dev = torch.from_numpy(rows).to(dev)
    q0 = to_bits(q[rows_dev])
    k0 = to_bits(k[rows_dev])
    cu_dev = torch.from_numpy(pack.cu_seqlens).to(dev)
    cache = pr().new_cos_sin_cache(T, w.head_dim, w.theta, device=dev)
    info = pr().rope_qk_launch_info(q, k, w.theta, cu_seqlens=cu_dev, cos_sin_cache=cache)
    assert info.kernel_name() == "rope_qk_tile_kernel<128,true,3>"          # 64-bit offsets, a cache: 3 units
    _run("rope_qk_fwd", q, k, cu_dev, w.theta, cache)
    pos = oracle.positions(pack.cu_seqlens, T)[rows]
    for x, y in ((q0, q), (k0, k)):
        s = compare(to_bits(y[rows_dev]), oracle.rope_rows(x, pos, w.theta), x)
        assert_parity(s, "w5 fwd")
        assert s["bit_mismatch"] == 0, s
    assert torch.equal(q_store[-guard:].view(torch.int16), canary.view(torch.int16))
    # backward on the rotated tensors brings the sampled rows back within rounding
    _run("rope_qk_bwd", q, k, cu_dev, w.theta, cache)
    for x, y in ((q0, q), (k0, k)):
        back = to_bits(y[rows_dev])
        ref = oracle.rope_rows(oracle.rope_rows(x, pos, w.theta), pos, w.theta, bwd=True)
        assert np.array_equal(back, ref)
    assert torch.equal(q_store[-guard:].view(torch.int16), canary.view(torch.int16))


@pytest.mark.parametrize("use_cache", [False, True])
def test_workload5_cp_rank_long_segments(dev, use_cache):
    """A load-balanced context-parallel rank of the 1,048,576-token sequence (cp = 2,
    rank 0: chunks 0 and 3 of 4): its 2^19 rows of 32 Q heads span 2^31 elements, so the
    64-bit-offset instance runs with a two-entry segment list whose second segment
    starts at token 786,432.  Seeded rows, the rows around the segment boundary and the
    last rows (which end at Q's flat offset 2^31) equal the oracle; a canary after Q
    survives."""
    from packed_varlen_rope_gb300 import cp_shards, shard_rows, shard_segments
    from packed_varlen_rope_gb300 import workloads as wl

    w = wl.WORKLOADS[5]
    pack = wl.make_pack(w)
    T = pack.total_tokens
    shards = cp_shards(T, 2, 0)
    segs = shard_segments(shards)
    n = len(shard_rows(shards))
    assert n == T // 2 and segs == [(0, 0), (T // 4, 3 * T // 4)]
    guard = 4096
    q_store = torch.empty(n * w.n_q_heads * w.head_dim + guard, dtype=torch.bfloat16, device=dev)
    q = q_store[: n * w.n_q_heads * w.head_dim].view(n, w.n_q_heads, w.head_dim)
    q.copy_(wl.normal_bf16((n, w.n_q_heads, w.head_dim), 5100, device="cuda"))
    canary = torch.full((guard,), -3.5, dtype=torch.bfloat16, device=dev)
    q_store[-guard:].copy_(canary)
    k = wl.normal_bf16((n, w.n_kv_heads, w.head_dim), 5200, device="cuda")
    cu_dev = torch.from_numpy(pack.cu_seqlens).to(dev)
    cache = pr().new_cos_sin_cache(T, w.head_dim, w.theta, device=dev) if use_cache else None
    info = pr().rope_qk_launch_info(q, k, w.theta, cu_seqlens=cu_dev, segments=segs, cos_sin_cache=cache)
    assert info.kernel_name() == "rope_qk_tile_kernel<128,true,%d>" % (3 if use_cache else 2)
    rng = np.random.Generator(np.random.PCG64(5300))
    cross = (1 << 31) // (w.n_q_heads * w.head_dim)
    fixed = [r for r in (0, 1, T // 4 - 1, T // 4, T // 4 + 1, cross - 2, cross - 1, cross, n - 1) if r < n]
    rows = np.unique(np.concatenate([rng.integers(0, n, 2048), fixed])).astype(np.int64)
    rows_dev = torch.from_numpy(rows).to(dev)
    q0, k0 = to_bits(q[rows_dev]), to_bits(k[rows_dev])
    pr().rope_qk_apply(q, k, w.theta, cu_seqlens=cu_dev, segments=segs, cos_sin_cache=cache)
    torch.cuda.synchronize()
    tokens = np.where(rows < T // 4, rows, rows - T // 4 + 3 * T // 4)
    pos = oracle.positions(pack.cu_seqlens, T)[tokens]
    for x, y in ((q0, q), (k0, k)):
        s = compare(to_bits(y[rows_dev]), oracle.rope_rows(x, pos, w.theta), x)
        assert_parity(s, "w5 cp rank")
        assert s["bit_mismatch"] == 0, s
    assert torch.equal(q_store[-guard:].view(torch.int16), canary.view(torch.int16))


# ------------------------------------------------------------------ edge cases

EDGE_PACKS = [
    # (lengths, extra tokens outside, n_q_heads, n_kv_heads, head_dim)
    ([1], 0, 1, 1, 16),
    ([3, 0, 5], 2, 3, 1, 32),
    ([17, 1, 1, 0, 40], 7, 5, 5, 48),
    ([100, 3, 77], 0, 7, 1, 64),
    ([33, 65], 13, 2, 2, 80),
    ([129, 0, 2], 1, 9, 3, 96),
    ([50, 61], 0, 4, 4, 112),
    ([31, 257, 2], 5, 16, 2, 128),
    ([45, 9], 3, 3, 2, 144),
    ([64], 9, 2, 1, 192),
    ([70, 1], 0, 3, 3, 240),
    ([40, 23], 4, 6, 2, 256),
    ([2000], 0, 64, 8, 128),
]


@pytest.mark.parametrize("case", range(len(EDGE_PACKS)))
@pytest.mark.parametrize("in_place", [True, False])
def test_edge_shapes(dev, case, in_place):
    lengths, extra, hq, hkv, d = EDGE_PACKS[case]
    rng = np.random.Generator(np.random.PCG64(100 + case))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1]) + extra
    theta = [1.0e4, 1.0e6, 5.0e5][case % 3]
    qb = _normal_bits(rng, (T, hq, d))
    kb = _normal_bits(rng, (T, hkv, d))
    q, k = from_bits(qb, dev), from_bits(kb, dev)
    cu_dev = torch.from_numpy(cu).to(dev)
    for bwd in (False, True):
        fn = "rope_qk_bwd" if bwd else "rope_qk_fwd"
        qi, ki = q.clone(), k.clone()
        if in_place:
            _run(fn, qi, ki, cu_dev, theta)
            qo, ko = qi, ki
        else:
            qo = torch.full_like(q, 3.0)
            ko = torch.full_like(k, 3.0)
            _run(fn, qi, ki, cu_dev, theta, in_place=False, q_out=qo, k_out=ko)
            assert torch.equal(qi.view(torch.int16), q.view(torch.int16))      # inputs only read
            assert torch.equal(ki.view(torch.int16), k.view(torch.int16))
        _check_full(qb, kb, cu, theta, qo, ko, bwd, (case, in_place, bwd))


def test_special_values(dev):
    rng = np.random.Generator(np.random.PCG64(40))
    specials = np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, -3.0e38, 1.0e-40, -1.0e-40, 2.0 ** -126, 65504.0,
                         1.0e30, -7.5e-39, 1.0 + 2.0 ** -7, 0.5], dtype=np.float32)
    T, H, d = 300, 3, 64
    vals = rng.choice(specials, size=(T, H, d)).astype(np.float32)
    bits = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    cu = np.array([0, 100, 299, 300], dtype=np.int32)
    kb = bits[:, :2].copy()
    for bwd in (False, True):
        q, k = from_bits(bits, dev), from_bits(kb, dev)
        _run("rope_qk_bwd" if bwd else "rope_qk_fwd", q, k, torch.from_numpy(cu).to(dev), 1.0e6)
        _check_full(bits, kb, cu, 1.0e6, q, k, bwd, ("special", bwd))


def test_cache_variants_identical(dev):
    """Full cache, partial cache (positions past its end evaluated on the fly) and no
    cache give the same bits."""
    w, pack, q, k, _, _ = _workload_inputs(2)
    cu_dev = torch.from_numpy(pack.cu_seqlens).to(dev)
    full = pr().new_cos_sin_cache(max(pack.lengths), w.head_dim, w.theta, device=dev)
    part = pr().new_cos_sin_cache(300, w.head_dim, w.theta, device=dev)
    outs = []
    for cache in (full, part, None):
        qi, ki = q.clone(), k.clone()
        _run("rope_qk_fwd", qi, ki, cu_dev, w.theta, cache)
        outs.append((qi.view(torch.int16), ki.view(torch.int16)))
    for o in outs[1:]:
        assert torch.equal(o[0], outs[0][0]) and torch.equal(o[1], outs[0][1])


def test_outside_tokens_and_empty(dev):
    rng = np.random.Generator(np.random.PCG64(41))
    T, hq, hkv, d = 50, 4, 2, 64
    qb, kb = _normal_bits(rng, (T, hq, d)), _normal_bits(rng, (T, hkv, d))
    for cu in ([0], [0, 0, 0], [5, 9, 20], [0, 50]):
        q, k = from_bits(qb, dev), from_bits(kb, dev)
        cu_np = np.array(cu, dtype=np.int32)
        _run("rope_qk_fwd", q, k, torch.from_numpy(cu_np).to(dev), 1.0e4)
        pos = oracle.positions(cu_np, T)
        outside = pos < 0
        assert np.array_equal(to_bits(q)[outside], qb[outside])
        assert np.array_equal(to_bits(q), oracle.rope_rows(qb, pos, 1.0e4))
    # an empty pack launches nothing and succeeds
    e = torch.empty((0, hq, d), dtype=torch.bfloat16, device=dev)
    ek = torch.empty((0, hkv, d), dtype=torch.bfloat16, device=dev)
    pr().rope_qk_fwd(e, ek, torch.zeros(1, dtype=torch.int32, device=dev), 1.0e4)


@pytest.mark.parametrize("with_seq_used", [False, True])
def test_invalid_cu_stays_in_bounds(dev, with_seq_used):
    """A decreasing cu_seqlens is reported by the validator; the rotation kernel still
    touches only rows of Q and K and leaves tokens outside [cu[0], cu[n]) alone (also
    with seq_used values beyond the samples' lengths and negative ones)."""
    rng = np.random.Generator(np.random.PCG64(42))
    T, hq, hkv, d = 64, 2, 1, 64
    guard = 2048
    store = torch.full((T * hq * d + 2 * guard,), 5.0, dtype=torch.bfloat16, device=dev)
    q = store[guard: guard + T * hq * d].view(T, hq, d)
    qb = _normal_bits(rng, (T, hq, d))
    q.copy_(from_bits(qb, dev))
    k = from_bits(_normal_bits(rng, (T, hkv, d)), dev)
    cu = torch.tensor([0, 40, 10, 30, 48], dtype=torch.int32, device=dev)
    assert int(pr().rope_validate_cu_seqlens(cu, T).item()) & pr().ROPE_CU_DECREASING
    if with_seq_used:
        used = torch.tensor([1000, -7, 12, 3], dtype=torch.int32, device=dev)
        pr().rope_qk_apply(q, k, 1.0e4, cu_seqlens=cu, seq_used=used)
        torch.cuda.synchronize()
    else:
        _run("rope_qk_fwd", q, k, cu, 1.0e4)
    assert torch.all(store[:guard] == 5.0) and torch.all(store[-guard:] == 5.0)
    assert np.array_equal(to_bits(q)[48:], qb[48:])


def test_guard_canaries(dev):
    from packed_varlen_rope_gb300 import workloads as wl

    w = wl.WORKLOADS[2]
    pack = wl.make_pack(w)
    T = pack.total_tokens
    guard = 4096
    nq, nk = T * w.n_q_heads * w.head_dim, T * w.n_kv_heads * w.head_dim
    store = torch.full((nq + nk + 3 * guard,), -2.5, dtype=torch.bfloat16, device=dev)
    q = store[guard: guard + nq].view(T, w.n_q_heads, w.head_dim)
    k = store[2 * guard + nq: 2 * guard + nq + nk].view(T, w.n_kv_heads, w.head_dim)
    q.normal_()
    k.normal_()
    cu_dev = torch.from_numpy(pack.cu_seqlens).to(dev)
    _run("rope_qk_fwd", q, k, cu_dev, w.theta)
    _run("rope_qk_bwd", q, k, cu_dev, w.theta)
    for sl in (slice(0, guard), slice(guard + nq, 2 * guard + nq), slice(2 * guard + nq + nk, None)):
        assert torch.all(store[sl] == -2.5)


def test_side_stream(dev):
    w, pack, q, k, _, _ = _workload_inputs(1)
    q0, k0 = to_bits(q), to_bits(k)
    cu_dev = torch.from_numpy(pack.cu_seqlens).to(dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pr().rope_qk_fwd(q, k, cu_dev, w.theta)
    s.synchronize()
    _check_full(q0, k0, pack.cu_seqlens, w.theta, q, k, False, "side stream")


def test_autograd(dev):
    from packed_varlen_rope_gb300 import apply_rope_qk

    w, pack, q, k, dq, dk = _workload_inputs(1)
    cu_dev = torch.from_numpy(pack.cu_seqlens).to(dev)
    q0, k0, g_q, g_k = (to_bits(t) for t in (q, k, dq, dk))
    qleaf = torch.zeros_like(q, requires_grad=True)
    kleaf = torch.zeros_like(k, requires_grad=True)
    qa = qleaf + q          # non-leaf copies that may be modified in place
    ka = kleaf + k
    yq, yk = apply_rope_qk(qa, ka, cu_dev, w.theta)
    torch.autograd.backward([yq, yk], [dq, dk])
    assert np.array_equal(to_bits(yq), oracle.rope_packed(q0, pack.cu_seqlens, w.theta))
    assert np.array_equal(to_bits(qleaf.grad), oracle.rope_packed(g_q, pack.cu_seqlens, w.theta, bwd=True))
    assert np.array_equal(to_bits(kleaf.grad), oracle.rope_packed(g_k, pack.cu_seqlens, w.theta, bwd=True))


def test_maximum_token_count(dev):
    """The largest pack the library takes: 2^24 tokens, so positions run to 2^24 - 1 (the
    last integer binary32 holds exactly) and the angles reach their largest values.  A
    small head shape keeps it to 1 GiB; sampled rows against the oracle, and one token
    more is refused."""
    T, hq, hkv, d = 1 << 24, 1, 1, 16
    q = torch.empty((T, hq, d), dtype=torch.bfloat16, device=dev).normal_()
    k = torch.empty((T, hkv, d), dtype=torch.bfloat16, device=dev).normal_()
    rng = np.random.Generator(np.random.PCG64(50))
    rows = np.unique(np.concatenate([rng.integers(0, T, 2000), [0, 1, T - 2, T - 1, (1 << 23), (1 << 23) + 1]]))
    rows_dev = torch.from_numpy(rows).to(dev)
    q0, k0 = to_bits(q[rows_dev]), to_bits(k[rows_dev])
    cu_np = np.array([0, T], dtype=np.int32)
    cu = torch.from_numpy(cu_np).to(dev)
    _run("rope_qk_fwd", q, k, cu, 1.0e6)
    pos = rows.astype(np.int32)
    for x, y in ((q0, q), (k0, k)):
        s = compare(to_bits(y[rows_dev]), oracle.rope_rows(x, pos, 1.0e6), x)
        assert_parity(s, "max T")
        assert s["bit_mismatch"] == 0, s
    over = torch.empty((T + 1, hq, d), dtype=torch.bfloat16, device=dev)
    with pytest.raises(pr().RopeError) as err:
        pr().rope_qk_fwd(over, torch.empty((T + 1, hkv, d), dtype=torch.bfloat16, device=dev),
                         torch.tensor([0, T + 1], dtype=torch.int32, device=dev), 1.0e6)
    assert err.value.status == -6


def test_rotary_embedding_module(dev):
    """RotaryEmbedding keeps a per-device cache sized from the host-known position bound:
    forward and backward equal the oracle (tiny pack) and the plain entry points (bit for
    bit, 16k pack), the cache grows to the next power of two when a longer pack comes,
    context-parallel halves with token_offset equal the whole pack, and a broadcast
    gradient (sum().backward()) is accepted."""
    from packed_varlen_rope_gb300 import RotaryEmbedding

    w, pack, q, k, dq, dk = _workload_inputs(1)
    cu_dev = torch.from_numpy(pack.cu_seqlens).to(dev)
    rope = RotaryEmbedding(w.head_dim, w.theta)
    q0, k0, g_q = (to_bits(t) for t in (q, k, dq))
    qleaf = torch.zeros_like(q, requires_grad=True)
    kleaf = torch.zeros_like(k, requires_grad=True)
    yq, yk = rope(qleaf + q, kleaf + k, cu_seqlens=cu_dev)
    torch.autograd.backward([yq, yk], [dq, dk])
    assert np.array_equal(to_bits(yq), oracle.rope_packed(q0, pack.cu_seqlens, w.theta))
    assert np.array_equal(to_bits(yk), oracle.rope_packed(k0, pack.cu_seqlens, w.theta))
    assert np.array_equal(to_bits(qleaf.grad), oracle.rope_packed(g_q, pack.cu_seqlens, w.theta, bwd=True))
    assert rope.cache(dev, 1).rows == 1024

    w2, pack2, q2, k2, dq2, dk2 = _workload_inputs(2)
    cu2 = torch.from_numpy(pack2.cu_seqlens).to(dev)
    rope2 = RotaryEmbedding(w2.head_dim, w2.theta)
    ref_q, ref_k = q2.clone(), k2.clone()
    pr().rope_qk_fwd(ref_q, ref_k, cu2, w2.theta)
    got_q, got_k = rope2(q2.clone(), k2.clone(), cu_seqlens=cu2)
    assert torch.equal(got_q, ref_q) and torch.equal(got_k, ref_k)
    assert rope2.cache(dev, 1).rows == 16384
    # two context-parallel halves of the same pack
    half = pack2.total_tokens // 2
    qa, ka = q2.clone(), k2.clone()
    rope2(qa[:half], ka[:half], cu_seqlens=cu2, token_offset=0)
    rope2(qa[half:], ka[half:], cu_seqlens=cu2, token_offset=half)
    assert torch.equal(qa, ref_q) and torch.equal(ka, ref_k)
    # a longer pack grows the cache
    T3 = 20000
    cu3 = torch.tensor([0, T3], dtype=torch.int32, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(31)
    q3 = torch.randn((T3, 2, w2.head_dim), device=dev, generator=gen).to(torch.bfloat16)
    k3 = torch.randn((T3, 1, w2.head_dim), device=dev, generator=gen).to(torch.bfloat16)
    ref3 = (q3.clone(), k3.clone())
    pr().rope_qk_fwd(ref3[0], ref3[1], cu3, w2.theta)
    out3 = rope2(q3, k3, cu_seqlens=cu3)
    assert rope2.cache(dev, 1).rows == 32768
    assert torch.equal(out3[0], ref3[0]) and torch.equal(out3[1], ref3[1])
    # broadcast gradient
    ql = torch.zeros((64, 2, w2.head_dim), dtype=torch.bfloat16, device=dev, requires_grad=True)
    kl = torch.zeros((64, 1, w2.head_dim), dtype=torch.bfloat16, device=dev, requires_grad=True)
    yq, yk = rope2(ql + 1, kl + 1, cu_seqlens=torch.tensor([0, 64], dtype=torch.int32, device=dev))
    (yq.float().sum() + yk.float().sum()).backward()
    ones = torch.ones((64, 2, w2.head_dim), dtype=torch.bfloat16, device=dev)
    expect = pr().rope_qk_bwd(ones.clone(), ones[:, :1].clone(), torch.tensor([0, 64], dtype=torch.int32,
                                                                               device=dev), w2.theta)
    assert torch.equal(ql.grad, expect[0]) and torch.equal(kl.grad, expect[1])


def test_rotary_embedding_cp_segments_autograd(dev):
    """RotaryEmbedding on a load-balanced context-parallel rank's buffer (cp = 2, rank 1:
    chunks 1 and 2 of 4) through its segment list: the forward equals the whole-pack
    rotation's rows and the autograd backward the oracle's transpose rotation, the cache
    grown to cover the rank's last global token."""
    from packed_varlen_rope_gb300 import RotaryEmbedding, cp_shards, shard_rows, shard_segments

    w, pack, q, k, dq, dk = _workload_inputs(2)
    T = pack.total_tokens
    cu_dev = torch.from_numpy(pack.cu_seqlens).to(dev)
    shards = cp_shards(T, 2, 1)
    rows = torch.tensor(shard_rows(shards), device=dev)
    assert int(rows.max()) < T
    rope = RotaryEmbedding(w.head_dim, w.theta)
    ql, kl = q[rows].clone(), k[rows].clone()
    g_q, g_k = dq[rows].clone(), dk[rows].clone()
    qleaf = torch.zeros_like(ql, requires_grad=True)
    kleaf = torch.zeros_like(kl, requires_grad=True)
    yq, yk = rope(qleaf + ql, kleaf + kl, cu_seqlens=cu_dev, segments=shard_segments(shards))
    torch.autograd.backward([yq, yk], [g_q, g_k])
    pos = oracle.positions(pack.cu_seqlens, T)[rows.cpu().numpy()]
    assert np.array_equal(to_bits(yq), oracle.rope_rows(to_bits(ql), pos, w.theta))
    assert np.array_equal(to_bits(yk), oracle.rope_rows(to_bits(kl), pos, w.theta))
    assert np.array_equal(to_bits(qleaf.grad), oracle.rope_rows(to_bits(g_q), pos, w.theta, bwd=True))
    assert np.array_equal(to_bits(kleaf.grad), oracle.rope_rows(to_bits(g_k), pos, w.theta, bwd=True))
    assert rope.cache(dev, 1).rows >= int(rows.max()) + 1


@pytest.mark.parametrize("use_cache", [True, False])
def test_rotary_embedding_seq_used_autograd(dev, use_cache):
    """RotaryEmbedding on the padded Llama-3-8B batch (8 x 2048 rows, 47 % valid) with
    seq_used: the forward rotates each sample's first seq_used[s] rows as the oracle does
    and leaves the pad rows' bits as they were; the autograd backward gives the oracle's
    transpose rotation on those rows and passes the pad rows' gradient through."""
    from packed_varlen_rope_gb300 import RotaryEmbedding

    w, pack, q, k, dq, dk = _workload_inputs(3, "padded")
    T = pack.total_tokens
    cu_dev = torch.from_numpy(pack.cu_seqlens).to(dev)
    used = torch.tensor(pack.lengths, dtype=torch.int32, device=dev)
    pos = oracle.positions(pack.cu_seqlens, T)
    sample = np.searchsorted(pack.cu_seqlens, np.arange(T), side="right") - 1
    valid = pos < np.asarray(pack.lengths)[sample]
    assert 0.4 < valid.mean() < 0.6
    rope = RotaryEmbedding(w.head_dim, w.theta, use_cache=use_cache)
    qleaf = torch.zeros_like(q, requires_grad=True)
    kleaf = torch.zeros_like(k, requires_grad=True)
    yq, yk = rope(qleaf + q, kleaf + k, cu_seqlens=cu_dev, seq_used=used)
    torch.autograd.backward([yq, yk], [dq, dk])
    for y, x, g, grad in ((yq, q, dq, qleaf.grad), (yk, k, dk, kleaf.grad)):
        xb, gb = to_bits(x), to_bits(g)
        yb, db = to_bits(y), to_bits(grad)
        assert np.array_equal(yb[valid], oracle.rope_rows(xb[valid], pos[valid], w.theta))
        assert np.array_equal(db[valid], oracle.rope_rows(gb[valid], pos[valid], w.theta, bwd=True))
        assert np.array_equal(yb[~valid], xb[~valid]) and np.array_equal(db[~valid], gb[~valid])


def test_rotary_embedding_without_cache(dev):
    """RotaryEmbedding(use_cache=False) builds no table and gives the bits of the cached
    module, forward and autograd backward."""
    from packed_varlen_rope_gb300 import RotaryEmbedding

    w, pack, q, k, dq, dk = _workload_inputs(2)
    cu_dev = torch.from_numpy(pack.cu_seqlens).to(dev)
    outs = []
    for use_cache in (True, False):
        rope = RotaryEmbedding(w.head_dim, w.theta, use_cache=use_cache)
        qleaf = torch.zeros_like(q, requires_grad=True)
        kleaf = torch.zeros_like(k, requires_grad=True)
        yq, yk = rope(qleaf + q, kleaf + k, cu_seqlens=cu_dev)
        torch.autograd.backward([yq, yk], [dq, dk])
        outs.append((yq.detach(), yk.detach(), qleaf.grad, kleaf.grad))
        assert (len(rope._caches) == 1) == use_cache
    for a, b in zip(*outs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_rotary_embedding_int64_position_ids(dev):
    """RotaryEmbedding with int64 position ids (a Hugging Face collator's dtype), forward
    and autograd backward, against the oracle on the same positions."""
    from packed_varlen_rope_gb300 import RotaryEmbedding

    w, pack, q, k, dq, dk = _workload_inputs(1)
    pos = oracle.positions(pack.cu_seqlens, pack.total_tokens).astype(np.int64)
    ids = torch.from_numpy(pos).to(dev)
    rope = RotaryEmbedding(w.head_dim, w.theta)
    q0, k0, g_q, g_k = (to_bits(t) for t in (q, k, dq, dk))
    qleaf = torch.zeros_like(q, requires_grad=True)
    kleaf = torch.zeros_like(k, requires_grad=True)
    yq, yk = rope(qleaf + q, kleaf + k, position_ids=ids)
    torch.autograd.backward([yq, yk], [dq, dk])
    p32 = pos.astype(np.int32)
    assert np.array_equal(to_bits(yq), oracle.rope_rows(q0, p32, w.theta))
    assert np.array_equal(to_bits(yk), oracle.rope_rows(k0, p32, w.theta))
    assert np.array_equal(to_bits(qleaf.grad), oracle.rope_rows(g_q, p32, w.theta, bwd=True))
    assert np.array_equal(to_bits(kleaf.grad), oracle.rope_rows(g_k, p32, w.theta, bwd=True))
    # global ids of a shard beyond its row count: the max_position hint sizes the cache
    big = torch.from_numpy(pos + 100_000).to(dev)
    qb = q.clone()
    rope(qb, k.clone(), position_ids=big, max_position=100_000 + int(pos.max()))
    assert rope.cache(dev, 1).rows >= 100_000 + int(pos.max()) + 1
    assert np.array_equal(to_bits(qb), oracle.rope_rows(q0, (pos + 100_000).astype(np.int32), w.theta))


def test_back_to_back_launches_see_previous_writes(dev):
    """Rotations are launched so that they may be scheduled while the previous kernel in
    the stream drains (programmatic dependent launch); they must still see everything
    that kernel wrote.  Q and K are rewritten right before each rotation by a torch
    conversion kernel, by a device copy, or by the previous rotation itself, 30 times in
    a row, and every result equals the oracle."""
    w, pack, q, k, dq, dk = _workload_inputs(2)
    cu = torch.from_numpy(pack.cu_seqlens).to(dev)
    cache = pr().new_cos_sin_cache(max(pack.lengths), w.head_dim, w.theta, device=dev)
    q0, k0 = to_bits(q), to_bits(k)
    once_q = oracle.rope_packed(q0, pack.cu_seqlens, w.theta)
    once_k = oracle.rope_packed(k0, pack.cu_seqlens, w.theta)
    twice_q = oracle.rope_packed(once_q, pack.cu_seqlens, w.theta)
    twice_k = oracle.rope_packed(once_k, pack.cu_seqlens, w.theta)
    qf, kf = q.float(), k.float()                    # exact: bf16 -> fp32 -> bf16
    qa, ka = torch.empty_like(q), torch.empty_like(k)
    for i in range(30):
        if i % 3 == 0:
            qa.copy_(qf)                             # conversion kernel
            ka.copy_(kf)
        else:
            qa.copy_(q)                              # same-dtype device copy
            ka.copy_(k)
        pr().rope_qk_fwd(qa, ka, cu, w.theta, cos_sin_cache=cache)
        if i % 2 == 1:
            pr().rope_qk_fwd(qa, ka, cu, w.theta, cos_sin_cache=cache)    # reads the previous rotation
        torch.cuda.synchronize()
        want_q, want_k = (twice_q, twice_k) if i % 2 == 1 else (once_q, once_k)
        assert np.array_equal(to_bits(qa), want_q) and np.array_equal(to_bits(ka), want_k), i
