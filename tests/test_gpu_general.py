"""The general entry point rope_qk_apply against the CPU oracle (needs a GB300).

Covers strided views (the Q and K slices of a fused QKV projection output rotated in
place, head-major layouts, strided outputs), explicit position ids, context-parallel
shards through a global token offset, and the linear position rescale.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from parity_util import assert_parity, compare, from_bits, to_bits

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


def _bits(rng, shape):
    f = torch.from_numpy(rng.standard_normal(size=shape).astype(np.float32))
    return f.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _pack(rng, n, max_len, extra=0):
    lengths = rng.integers(0, max_len + 1, size=n)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return cu, int(cu[-1]) + extra


def _expect(x_bits, pos, theta, bwd=False, scale=1.0):
    return oracle.rope_rows(x_bits, pos, theta, bwd=bwd, scale=scale)


def _check(got_bits, ref_bits, x_bits, what):
    s = compare(got_bits, ref_bits, x_bits)
    assert_parity(s, what)
    assert s["bit_mismatch"] == 0, (what, s)


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 128), (4, 2, 64), (6, 1, 96), (8, 8, 256)])
@pytest.mark.parametrize("bwd", [False, True])
def test_fused_qkv_in_place(dev, hq, hkv, d, bwd):
    rng = np.random.Generator(np.random.PCG64(hq * 1000 + d))
    cu, T = _pack(rng, 9, 300, extra=5)
    qkv_bits = _bits(rng, (T, hq + 2 * hkv, d))
    qkv = from_bits(qkv_bits, dev)
    q, k = qkv[:, :hq], qkv[:, hq:hq + hkv]
    pr().rope_qk_apply(q, k, 1.0e6, cu_seqlens=torch.from_numpy(cu).to(dev), backward=bwd)
    torch.cuda.synchronize()
    out = to_bits(qkv)
    pos = oracle.positions(cu, T)
    _check(out[:, :hq], _expect(qkv_bits[:, :hq], pos, 1.0e6, bwd), qkv_bits[:, :hq], "fused q")
    _check(out[:, hq:hq + hkv], _expect(qkv_bits[:, hq:hq + hkv], pos, 1.0e6, bwd),
           qkv_bits[:, hq:hq + hkv], "fused k")
    assert np.array_equal(out[:, hq + hkv:], qkv_bits[:, hq + hkv:])          # V untouched


def test_fused_qkv_workload2_with_cache(dev):
    """Qwen3-4B shape, 16,384 packed tokens, rotated inside its fused QKV buffer."""
    from packed_varlen_rope_gb300 import workloads as wl

    w = wl.WORKLOADS[2]
    pack = wl.make_pack(w)
    T, hq, hkv, d = pack.total_tokens, w.n_q_heads, w.n_kv_heads, w.head_dim
    qkv = wl.normal_bf16((T, hq + 2 * hkv, d), 91, device="cuda")
    before = to_bits(qkv)
    cache = pr().new_cos_sin_cache(max(pack.lengths), d, w.theta, device=dev)
    pr().rope_qk_apply(qkv[:, :hq], qkv[:, hq:hq + hkv], w.theta,
                       cu_seqlens=torch.from_numpy(pack.cu_seqlens).to(dev), cos_sin_cache=cache)
    torch.cuda.synchronize()
    out = to_bits(qkv)
    pos = oracle.positions(pack.cu_seqlens, T)
    for sl in (slice(0, hq), slice(hq, hq + hkv)):
        _check(out[:, sl], _expect(before[:, sl], pos, w.theta), before[:, sl], "w2 fused")
    assert np.array_equal(out[:, hq + hkv:], before[:, hq + hkv:])


def test_head_major_views(dev):
    """Q stored [H, T, d] (a transposed view): token stride d, head stride T*d."""
    rng = np.random.Generator(np.random.PCG64(5))
    cu, T = _pack(rng, 6, 200)
    hq, hkv, d = 5, 3, 64
    qb = _bits(rng, (hq, T, d))
    kb = _bits(rng, (hkv, T, d))
    qh, kh = from_bits(qb, dev), from_bits(kb, dev)
    pr().rope_qk_apply(qh.permute(1, 0, 2), kh.permute(1, 0, 2), 1.0e4,
                       cu_seqlens=torch.from_numpy(cu).to(dev))
    torch.cuda.synchronize()
    pos = oracle.positions(cu, T)
    q_tok = np.ascontiguousarray(qb.transpose(1, 0, 2))
    k_tok = np.ascontiguousarray(kb.transpose(1, 0, 2))
    _check(np.ascontiguousarray(to_bits(qh).transpose(1, 0, 2)), _expect(q_tok, pos, 1.0e4), q_tok, "hm q")
    _check(np.ascontiguousarray(to_bits(kh).transpose(1, 0, 2)), _expect(k_tok, pos, 1.0e4), k_tok, "hm k")


def test_out_of_place_into_fused_buffer(dev):
    rng = np.random.Generator(np.random.PCG64(6))
    cu, T = _pack(rng, 5, 150, extra=3)
    hq, hkv, d = 4, 2, 128
    qb, kb = _bits(rng, (T, hq, d)), _bits(rng, (T, hkv, d))
    q, k = from_bits(qb, dev), from_bits(kb, dev)
    out = torch.full((T, hq + 2 * hkv, d), 9.0, dtype=torch.bfloat16, device=dev)
    pr().rope_qk_apply(q, k, 5.0e5, cu_seqlens=torch.from_numpy(cu).to(dev),
                       q_out=out[:, :hq], k_out=out[:, hq:hq + hkv])
    torch.cuda.synchronize()
    pos = oracle.positions(cu, T)
    ob = to_bits(out)
    _check(ob[:, :hq], _expect(qb, pos, 5.0e5), qb, "ooq")
    _check(ob[:, hq:hq + hkv], _expect(kb, pos, 5.0e5), kb, "ook")
    assert torch.all(out[:, hq + hkv:] == 9.0)
    assert np.array_equal(to_bits(q), qb) and np.array_equal(to_bits(k), kb)


def test_position_ids_equal_cu_path(dev):
    from packed_varlen_rope_gb300 import workloads as wl

    w = wl.WORKLOADS[3]
    pack = wl.make_pack(w, "padded")
    T = pack.total_tokens
    q = wl.normal_bf16((T, w.n_q_heads, w.head_dim), 3, device="cuda")
    k = wl.normal_bf16((T, w.n_kv_heads, w.head_dim), 4, device="cuda")
    q2, k2 = q.clone(), k.clone()
    cu = torch.from_numpy(pack.cu_seqlens).to(dev)
    pr().rope_qk_fwd(q, k, cu, w.theta)
    pos = pr().rope_qk_positions(cu, T)
    pr().rope_qk_apply(q2, k2, w.theta, position_ids=pos)
    torch.cuda.synchronize()
    assert torch.equal(q.view(torch.int16), q2.view(torch.int16))
    assert torch.equal(k.view(torch.int16), k2.view(torch.int16))


@pytest.mark.parametrize("dtype", ["int32", "int64"])
def test_position_ids_arbitrary(dev, dtype):
    """Explicit ids in any order, including ids outside [0, 2^24) which leave the row out;
    int64 ids (ROPE_FLAG_POSITION_IDS_INT64) also with values beyond the int32 range."""
    rng = np.random.Generator(np.random.PCG64(7))
    T, hq, hkv, d = 300, 3, 2, 64
    ids = rng.integers(0, 1 << 24, size=T).astype(np.int64)
    ids[:10] = [0, 1, (1 << 24) - 1, -1, -7, 1 << 24, (1 << 31) - 1, 5, 100000, 25000]
    if dtype == "int64":
        ids[10:15] = [1 << 33, -(1 << 40), (1 << 62), (1 << 32) + 5, -(1 << 63)]
    ids_np = ids.astype(np.int32 if dtype == "int32" else np.int64)
    qb, kb = _bits(rng, (T, hq, d)), _bits(rng, (T, hkv, d))
    for bwd in (False, True):
        q, k = from_bits(qb, dev), from_bits(kb, dev)
        pid = torch.from_numpy(ids_np).to(dev)
        pr().rope_qk_apply(q, k, 1.0e6, position_ids=pid, backward=bwd)
        torch.cuda.synchronize()
        v = ids_np.astype(np.int64)
        pos = np.where((v >= 0) & (v < (1 << 24)), v, -1).astype(np.int32)
        _check(to_bits(q), _expect(qb, pos, 1.0e6, bwd), qb, "ids q")
        _check(to_bits(k), _expect(kb, pos, 1.0e6, bwd), kb, "ids k")


@pytest.mark.parametrize("cp", [2, 4])
def test_context_parallel_shards(dev, cp):
    """Shards of one pack, each holding its tokens and the pack's cu_seqlens with its
    token offset, give the unsharded result.  Both the contiguous split and the
    load-balanced split into 2*cp chunks (rank r holds chunks r and 2*cp-1-r) of the
    TRL context-parallel section are covered."""
    from packed_varlen_rope_gb300 import workloads as wl

    w = wl.WORKLOADS[2]
    pack = wl.make_pack(w)
    T = pack.total_tokens
    cu = torch.from_numpy(pack.cu_seqlens).to(dev)
    q = wl.normal_bf16((T, w.n_q_heads, w.head_dim), 8, device="cuda")
    k = wl.normal_bf16((T, w.n_kv_heads, w.head_dim), 9, device="cuda")
    q0, k0 = to_bits(q), to_bits(k)
    ref_q, ref_k = q.clone(), k.clone()
    pr().rope_qk_fwd(ref_q, ref_k, cu, w.theta)
    n_chunks = 2 * cp
    bounds = np.linspace(0, T, n_chunks + 1).astype(np.int64)
    layouts = {
        "contiguous": [[(int(bounds[2 * r]), int(bounds[2 * r + 2]))] for r in range(cp)],
        "balanced": [[(int(bounds[r]), int(bounds[r + 1])), (int(bounds[n_chunks - 1 - r]), int(bounds[n_chunks - r]))]
                     for r in range(cp)],
    }
    for name, ranks in layouts.items():
        out_q, out_k = torch.empty_like(q), torch.empty_like(k)
        for chunks in ranks:
            for a, b in chunks:
                sq, sk = q[a:b].clone(), k[a:b].clone()            # the shard's own buffers
                pr().rope_qk_apply(sq, sk, w.theta, cu_seqlens=cu, token_offset=a)
                out_q[a:b], out_k[a:b] = sq, sk
        torch.cuda.synchronize()
        assert torch.equal(out_q.view(torch.int16), ref_q.view(torch.int16)), name
        assert torch.equal(out_k.view(torch.int16), ref_k.view(torch.int16)), name
    pos = oracle.positions(pack.cu_seqlens, T)
    _check(to_bits(ref_k), _expect(k0, pos, w.theta), k0, "cp ref k")


@pytest.mark.parametrize("idx,cp", [(2, 2), (2, 4), (3, 3)])
@pytest.mark.parametrize("bwd", [False, True])
def test_cp_ranks_one_launch_each(dev, idx, cp, bwd):
    """Load-balanced context parallelism with the package's shard plan: each rank's
    buffer holds its two chunks (padding included) and is rotated in ONE launch through
    the segment list; put back in pack order, the ranks' rows equal the oracle over the
    whole pack bit for bit, and the padding rows are untouched."""
    from packed_varlen_rope_gb300 import workloads as wl

    w = wl.WORKLOADS[idx]
    pack = wl.make_pack(w)
    T = pack.total_tokens
    cu = torch.from_numpy(pack.cu_seqlens).to(dev)
    q = wl.normal_bf16((T, w.n_q_heads, w.head_dim), 18, device="cuda")
    k = wl.normal_bf16((T, w.n_kv_heads, w.head_dim), 19, device="cuda")
    q0, k0 = to_bits(q), to_bits(k)
    cache = pr().new_cos_sin_cache(max(pack.lengths), w.head_dim, w.theta, device=dev)
    got_q, got_k = np.zeros_like(q0), np.zeros_like(k0)
    seen = np.zeros(T, dtype=np.int32)
    for r in range(cp):
        shards = pr().cp_shards(T, cp, r, load_balanced=True)
        rows = np.array(pr().shard_rows(shards))
        inside = rows < T
        lq = np.full((rows.size,) + q0.shape[1:], 0x4040, np.uint16)        # padding rows: 3.0
        lk = np.full((rows.size,) + k0.shape[1:], 0x4040, np.uint16)
        lq[inside], lk[inside] = q0[rows[inside]], k0[rows[inside]]
        dq, dk = from_bits(lq, dev), from_bits(lk, dev)
        info = pr().rope_qk_launch_info(dq, dk, w.theta, cu_seqlens=cu, segments=pr().shard_segments(shards),
                                        cos_sin_cache=cache, backward=bwd)
        assert info.grid == -(-rows.size // info.tile_tokens)              # one launch covers the rank
        pr().rope_qk_apply(dq, dk, w.theta, cu_seqlens=cu, segments=pr().shard_segments(shards),
                           cos_sin_cache=cache, backward=bwd)
        torch.cuda.synchronize()
        oq, ok = to_bits(dq), to_bits(dk)
        assert np.all(oq[~inside] == 0x4040) and np.all(ok[~inside] == 0x4040)
        got_q[rows[inside]], got_k[rows[inside]] = oq[inside], ok[inside]
        seen[rows[inside]] += 1
    assert np.all(seen == 1)
    _check(got_q, oracle.rope_packed(q0, pack.cu_seqlens, w.theta, bwd=bwd), q0, ("cp q", idx, cp))
    _check(got_k, oracle.rope_packed(k0, pack.cu_seqlens, w.theta, bwd=bwd), k0, ("cp k", idx, cp))


@pytest.mark.parametrize("sp", [4, 16])
def test_ulysses_head_shards(dev, sp):
    """Ulysses sequence parallelism on the Qwen3-32B head shape (64 Q / 8 K heads): each
    rank holds every token of its heads (sp = 4: 16 Q and 2 K heads; sp = 16: 4 Q heads
    and the one K head they share) and rotates them alone; each rank's result equals the
    same heads of the whole rotation, which equals the oracle."""
    from packed_varlen_rope_gb300 import ulysses_heads
    from packed_varlen_rope_gb300 import workloads as wl

    w = wl.WORKLOADS[2]
    pack = wl.make_pack(w)
    T, hq, hkv, d = pack.total_tokens, 64, 8, w.head_dim
    cu = torch.from_numpy(pack.cu_seqlens).to(dev)
    q = wl.normal_bf16((T, hq, d), 71, device=dev)
    k = wl.normal_bf16((T, hkv, d), 72, device=dev)
    ref_q, ref_k = q.clone(), k.clone()
    pr().rope_qk_fwd(ref_q, ref_k, cu, w.theta)
    for r in range(sp):
        (q0, q1), (k0, k1) = ulysses_heads(hq, hkv, sp, r)
        ql, kl = q[:, q0:q1].contiguous(), k[:, k0:k1].contiguous()      # the rank's own buffers
        pr().rope_qk_fwd(ql, kl, cu, w.theta)
        assert torch.equal(ql, ref_q[:, q0:q1]) and torch.equal(kl, ref_k[:, k0:k1]), r
    pos = oracle.positions(pack.cu_seqlens, T)
    kb = to_bits(k)
    _check(to_bits(ref_k), _expect(kb, pos, w.theta), kb, "ulysses ref k")


def test_position_scale_page_example(dev):
    """TRL YaRN section: with factor 4, position 100,000 reads as 25,000 (and 163,840
    as 40,960) -- bit-identical rows, with and without a cos/sin cache."""
    rng = np.random.Generator(np.random.PCG64(10))
    hq, hkv, d = 4, 2, 128
    xb, kb = _bits(rng, (2, hq, d)), _bits(rng, (2, hkv, d))
    for use_cache in (False, True):
        outs = []
        for ids, scale in (([100000, 163840], 4.0), ([25000, 40960], 1.0)):
            q, k = from_bits(xb, dev), from_bits(kb, dev)
            cache = None
            if use_cache:
                cache = pr().new_cos_sin_cache(163841, d, 1.0e6, device=dev, position_scale=scale)
            pr().rope_qk_apply(q, k, 1.0e6, position_ids=torch.tensor(ids, dtype=torch.int32, device=dev),
                               position_scale=scale, cos_sin_cache=cache)
            torch.cuda.synchronize()
            outs.append((to_bits(q), to_bits(k)))
        assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("scale", [4.0, 2.5])
def test_position_scale_parity(dev, scale):
    from packed_varlen_rope_gb300 import workloads as wl

    w = wl.WORKLOADS[2]
    pack = wl.make_pack(w)
    T = pack.total_tokens
    q = wl.normal_bf16((T, w.n_q_heads, w.head_dim), 11, device="cuda")
    k = wl.normal_bf16((T, w.n_kv_heads, w.head_dim), 12, device="cuda")
    q0, k0 = to_bits(q), to_bits(k)
    cache = pr().new_cos_sin_cache(max(pack.lengths), w.head_dim, w.theta, device=dev, position_scale=scale)
    cu = torch.from_numpy(pack.cu_seqlens).to(dev)
    pr().rope_qk_apply(q, k, w.theta, cu_seqlens=cu, position_scale=scale, cos_sin_cache=cache)
    torch.cuda.synchronize()
    pos = oracle.positions(pack.cu_seqlens, T)
    _check(to_bits(q), _expect(q0, pos, w.theta, scale=scale), q0, "scaled q")
    _check(to_bits(k), _expect(k0, pos, w.theta, scale=scale), k0, "scaled k")
    # the scaled cache holds the oracle's scaled cos/sin
    host = pr()._binding.cache_as_cos_sin(cache.data[:64].cpu().numpy())
    for p in range(64):
        c, s = oracle.cos_sin(p, w.theta, w.head_dim, scale)
        assert np.array_equal(host[p, :, 0], c) and np.array_equal(host[p, :, 1], s)


def test_long_strided_fused_qkv(dev):
    """A fused QKV buffer of 2^20 tokens x (32 + 2*8) heads x 128 (6.4e9 elements): the
    Q/K views span more than 2^31 elements, so the 64-bit-offset kernel runs on strided
    views.  Sampled rows around the 2^31 element offset against the oracle."""
    T, hq, hkv, d = 1 << 20, 32, 8, 128
    from packed_varlen_rope_gb300 import workloads as wl

    qkv = wl.normal_bf16((T, hq + 2 * hkv, d), 13, device="cuda")
    per_token = (hq + 2 * hkv) * d
    cross = (1 << 31) // per_token
    rng = np.random.Generator(np.random.PCG64(14))
    rows = np.unique(np.concatenate([rng.integers(0, T, 512), [0, cross - 1, cross, cross + 1, T - 1]]))
    rows_dev = torch.from_numpy(rows).to(dev)
    before = to_bits(qkv[rows_dev])
    cu = torch.tensor([0, 300000, T], dtype=torch.int32, device=dev)
    pr().rope_qk_apply(qkv[:, :hq], qkv[:, hq:hq + hkv], 1.0e6, cu_seqlens=cu)
    torch.cuda.synchronize()
    after = to_bits(qkv[rows_dev])
    pos = oracle.positions(np.array([0, 300000, T], dtype=np.int32), T)[rows]
    for sl in (slice(0, hq), slice(hq, hq + hkv)):
        _check(after[:, sl], _expect(before[:, sl], pos, 1.0e6), before[:, sl], "long fused")
    assert np.array_equal(after[:, hq + hkv:], before[:, hq + hkv:])


def test_seq_used_skips_padding(dev):
    """Llama-3-8B shape padded to 8 x 2048 with uniform cu_seqlens and seq_used = the
    samples' lengths: pad rows are not touched, valid rows equal the packed run."""
    from packed_varlen_rope_gb300 import workloads as wl

    w = wl.WORKLOADS[3]
    padded, packed = wl.make_pack(w, "padded"), wl.make_pack(w, "packed")
    T = padded.total_tokens
    q = wl.normal_bf16((T, w.n_q_heads, w.head_dim), 31, device="cuda")
    k = wl.normal_bf16((T, w.n_kv_heads, w.head_dim), 32, device="cuda")
    q0, k0 = to_bits(q), to_bits(k)
    used = torch.tensor(padded.lengths, dtype=torch.int32, device=dev)
    pr().rope_qk_apply(q, k, w.theta, cu_seqlens=torch.from_numpy(padded.cu_seqlens).to(dev), seq_used=used)
    torch.cuda.synchronize()
    valid = padded.valid_mask
    pos = np.where(valid, oracle.positions(padded.cu_seqlens, T), -1).astype(np.int32)
    _check(to_bits(q), _expect(q0, pos, w.theta), q0, "seq_used q")
    _check(to_bits(k), _expect(k0, pos, w.theta), k0, "seq_used k")
    assert np.array_equal(to_bits(q)[~valid], q0[~valid])
    # the valid rows are the packed run's rows
    qp, kp = torch.from_numpy(q0[valid].view(np.int16)).view(torch.bfloat16).to(dev), \
        torch.from_numpy(k0[valid].view(np.int16)).view(torch.bfloat16).to(dev)
    pr().rope_qk_fwd(qp, kp, torch.from_numpy(packed.cu_seqlens).to(dev), w.theta)
    torch.cuda.synchronize()
    assert np.array_equal(to_bits(qp), to_bits(q)[valid])


@pytest.mark.parametrize("T,hq,hkv,d,cached,used,kernel,tile", [
    (32767, 32, 8, 128, True, False, "rope_qk_tile_kernel<128,false,3>", 1),    # short: 1-token tiles, 3 units
    (32768, 32, 8, 128, True, False, "rope_qk_tile_kernel<128,false,2>", 2),    # 2-token tiles, 2 units
    (32767, 64, 8, 128, True, False, "rope_qk_tile_kernel<128,false,2>", 1),    # 576 units: one batch of 3 won't hold
    (32768, 64, 8, 128, True, False, "rope_qk_tile_kernel<128,false,4>", 1),    # wide: 4 units
    (9001, 32, 8, 128, False, False, "rope_qk_tile_kernel<128,false,2>", 2),    # no cache
    (9001, 32, 8, 128, True, True, "rope_qk_tile_kernel<128,false,2>", 4),      # seq_used: 4-token tiles
    (5003, 4, 2, 64, True, False, "rope_qk_tile_kernel<64,false,3>", 11),       # small heads: 11-token tiles
    (5003, 6, 2, 80, True, False, "rope_qk_tile_kernel<0,false,2>", 7),         # generic head_dim
])
def test_dispatch_boundaries(dev, T, hq, hkv, d, cached, used, kernel, tile):
    """Each tile size and unroll the launch plan picks, at and just below the 32,768-tile
    edge and on ragged tails, forward and backward: every row equals the oracle (rows
    past a sample's seq_used, and past the pack's end, left as they were)."""
    rng = np.random.Generator(np.random.PCG64(T * 131 + hq * 7 + d))
    lengths = list(rng.integers(1, 3000, size=64))
    while sum(lengths) < T:
        lengths += list(rng.integers(1, 3000, size=64))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    n = int(np.searchsorted(cu, T - 3))          # the last sample ends 3 rows before T:
    cu = np.concatenate([cu[:n], [T - 3]]).astype(np.int32)   # rows past the pack stay as they are
    seq_used = None
    pos = oracle.positions(cu, T)
    if used:
        lens = np.diff(cu)
        use = np.floor(rng.random(lens.size) * (lens + 1)).astype(np.int32)    # uniform in [0, len]
        seq_used = torch.from_numpy(use).to(dev)
        sample = np.clip(np.searchsorted(cu, np.arange(T), side="right") - 1, 0, lens.size - 1)
        pos = np.where((pos >= 0) & (pos < use[sample]), pos, -1).astype(np.int32)
    cu_dev = torch.from_numpy(cu).to(dev)
    cache = pr().new_cos_sin_cache(int(np.diff(cu).max()), d, 1.0e6, device=dev) if cached else None
    qb, kb = _bits(rng, (T, hq, d)), _bits(rng, (T, hkv, d))
    for bwd in (False, True):
        q, k = from_bits(qb, dev), from_bits(kb, dev)
        info = pr().rope_qk_launch_info(q, k, 1.0e6, cu_seqlens=cu_dev, cos_sin_cache=cache, seq_used=seq_used)
        assert (info.kernel_name(), info.tile_tokens) == (kernel, tile)
        pr().rope_qk_apply(q, k, 1.0e6, cu_seqlens=cu_dev, cos_sin_cache=cache, seq_used=seq_used, backward=bwd)
        torch.cuda.synchronize()
        _check(to_bits(q), _expect(qb, pos, 1.0e6, bwd=bwd), qb, (kernel, "q", bwd))
        _check(to_bits(k), _expect(kb, pos, 1.0e6, bwd=bwd), kb, (kernel, "k", bwd))


@pytest.mark.parametrize("use_cache", [False, True])
def test_largest_pack(dev, use_cache):
    """The largest pack the library takes: 2^24 tokens in one sample (every position an
    exact binary32 integer up to 16,777,215), one Q and one K head of 16.  Seeded rows
    and the last rows equal the oracle, forward and backward; with the 2^24-row cos/sin
    cache or without one (the largest angles then go to the binary64 evaluation)."""
    T, d, theta = 1 << 24, 16, 1.0e4
    rng = np.random.Generator(np.random.PCG64(77))
    cu_np = np.array([0, T], dtype=np.int32)
    cu = torch.from_numpy(cu_np).to(dev)
    q = torch.empty((T, 1, d), dtype=torch.bfloat16, device=dev).normal_(generator=torch.Generator(dev).manual_seed(78))
    k = torch.empty((T, 1, d), dtype=torch.bfloat16, device=dev).normal_(generator=torch.Generator(dev).manual_seed(79))
    rows = np.unique(np.concatenate([rng.integers(0, T, 4096), np.arange(T - 40, T), [0, 1, 1 << 23]]))
    rows_dev = torch.from_numpy(rows).to(dev)
    q0, k0 = to_bits(q[rows_dev]), to_bits(k[rows_dev])
    cache = pr().new_cos_sin_cache(T, d, theta, device=dev) if use_cache else None
    pos = rows.astype(np.int32)
    for bwd in (False, True):
        pr().rope_qk_apply(q, k, theta, cu_seqlens=cu, cos_sin_cache=cache, backward=bwd)
        torch.cuda.synchronize()
        q0 = _expect(q0, pos, theta, bwd=bwd)
        k0 = _expect(k0, pos, theta, bwd=bwd)
        assert np.array_equal(to_bits(q[rows_dev]), q0) and np.array_equal(to_bits(k[rows_dev]), k0), bwd
