"""rope_qk_host: Q and K in host memory, streamed through a device workspace in chunks
(needs a GB300).  The result must be bit-identical to the device path and to the
oracle, whatever the chunking."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from parity_util import assert_parity, compare, to_bits

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


def _inputs(idx):
    from packed_varlen_rope_gb300 import workloads as wl

    w = wl.WORKLOADS[idx]
    pack = wl.make_pack(w)
    T = pack.total_tokens
    q = wl.normal_bf16((T, w.n_q_heads, w.head_dim), wl.seed(idx, "q"), device="cpu")
    k = wl.normal_bf16((T, w.n_kv_heads, w.head_dim), wl.seed(idx, "k"), device="cpu")
    return w, pack, q, k


def _workspace(dev, tokens, w):
    per_token = (w.n_q_heads + w.n_kv_heads) * w.head_dim * 2
    return torch.empty(2 * tokens * per_token + 4096, dtype=torch.uint8, device=dev)


@pytest.mark.parametrize("chunk_tokens", [8, 504, 4096, 20000])
@pytest.mark.parametrize("bwd", [False, True])
def test_host_stream_equals_device(dev, chunk_tokens, bwd):
    w, pack, q, k = _inputs(2)
    cu = torch.from_numpy(pack.cu_seqlens).to(dev)
    cache = pr().new_cos_sin_cache(max(pack.lengths), w.head_dim, w.theta, device=dev)
    qd, kd = q.to(dev), k.to(dev)
    (pr().rope_qk_bwd if bwd else pr().rope_qk_fwd)(qd, kd, cu, w.theta, cos_sin_cache=cache)
    qh, kh = q.clone().pin_memory(), k.clone().pin_memory()
    ws = _workspace(dev, chunk_tokens, w)
    pr().rope_qk_host(qh, kh, w.theta, ws, cu_seqlens=cu, backward=bwd, cos_sin_cache=cache)
    torch.cuda.current_stream(dev).synchronize()
    assert torch.equal(qh.view(torch.int16), qd.cpu().view(torch.int16))
    assert torch.equal(kh.view(torch.int16), kd.cpu().view(torch.int16))
    if chunk_tokens == 504 and not bwd:
        pos = oracle.positions(pack.cu_seqlens, pack.total_tokens)
        for x, y in ((q, qh), (k, kh)):
            xb = to_bits(x)
            s = compare(to_bits(y), oracle.rope_rows(xb, pos, w.theta), xb)
            assert_parity(s, "host stream")
            assert s["bit_mismatch"] == 0


def test_host_stream_out_of_place_ids_and_pageable(dev):
    w, pack, q, k = _inputs(3)
    pos = torch.from_numpy(oracle.positions(pack.cu_seqlens, pack.total_tokens)).to(dev)
    ref_q, ref_k = q.to(dev), k.to(dev)
    pr().rope_qk_apply(ref_q, ref_k, w.theta, position_ids=pos)
    qo, ko = torch.full_like(q, 2.0), torch.full_like(k, 2.0)          # pageable host outputs
    q_in, k_in = q.clone(), k.clone()
    pr().rope_qk_host(q_in, k_in, w.theta, _workspace(dev, 96, w), position_ids=pos, q_out=qo, k_out=ko)
    torch.cuda.current_stream(dev).synchronize()
    assert torch.equal(qo.view(torch.int16), ref_q.cpu().view(torch.int16))
    assert torch.equal(ko.view(torch.int16), ref_k.cpu().view(torch.int16))
    assert torch.equal(q_in.view(torch.int16), q.view(torch.int16))   # inputs untouched
    # the same with int64 ids: each chunk must read its own slice of the 8-byte ids
    qo64, ko64 = torch.full_like(q, 2.0), torch.full_like(k, 2.0)
    pr().rope_qk_host(q_in, k_in, w.theta, _workspace(dev, 96, w), position_ids=pos.to(torch.int64),
                      q_out=qo64, k_out=ko64)
    torch.cuda.current_stream(dev).synchronize()
    assert torch.equal(qo64.view(torch.int16), qo.view(torch.int16))
    assert torch.equal(ko64.view(torch.int16), ko.view(torch.int16))


def test_host_stream_token_offset(dev):
    """A context-parallel shard held on the host: tokens [a, b) with the pack's
    cu_seqlens and token_offset = a."""
    w, pack, q, k = _inputs(2)
    cu = torch.from_numpy(pack.cu_seqlens).to(dev)
    ref_q, ref_k = q.to(dev), k.to(dev)
    pr().rope_qk_fwd(ref_q, ref_k, cu, w.theta)
    a, b = 5000, 11000
    sq, sk = q[a:b].clone().pin_memory(), k[a:b].clone().pin_memory()
    pr().rope_qk_host(sq, sk, w.theta, _workspace(dev, 1000, w), cu_seqlens=cu, token_offset=a)
    torch.cuda.current_stream(dev).synchronize()
    assert torch.equal(sq.view(torch.int16), ref_q[a:b].cpu().view(torch.int16))
    assert torch.equal(sk.view(torch.int16), ref_k[a:b].cpu().view(torch.int16))


def test_host_stream_rejects_small_workspace(dev):
    w, pack, q, k = _inputs(1)
    cu = torch.from_numpy(pack.cu_seqlens).to(dev)
    with pytest.raises(pr().RopeError) as err:
        pr().rope_qk_host(q, k, w.theta, _workspace(dev, 1, w)[:512], cu_seqlens=cu)
    assert err.value.status == -6


@pytest.mark.parametrize("static", [False, True])
def test_host_call_rejected_late_leaves_buffers_untouched(dev, static):
    """A pack whose global token indices pass 2^24 only in its last chunk: both host
    entry points reject it before the first copy, so the caller's host buffers keep
    their contents (no chunk was rotated and copied back)."""
    w, pack, q, k = _inputs(2)
    cu = torch.from_numpy(pack.cu_seqlens).to(dev)
    qh, kh = q.clone().pin_memory(), k.clone().pin_memory()
    offset = (1 << 24) - pack.total_tokens + 1
    ws = None if static else _workspace(dev, 504, w)
    with pytest.raises(pr().RopeError) as err:
        pr().rope_qk_host(qh, kh, w.theta, ws, cu_seqlens=cu, token_offset=offset, device=dev)
    assert err.value.status == -6
    cache = pr().new_cos_sin_cache(64, w.head_dim, w.theta * 2, device=dev)     # built for another theta
    with pytest.raises(pr().RopeError) as err:
        pr().rope_qk_host(qh, kh, w.theta, ws, cu_seqlens=cu, cos_sin_cache=cache, device=dev)
    assert err.value.status == -11
    torch.cuda.synchronize()
    assert torch.equal(qh.view(torch.int16), q.view(torch.int16))
    assert torch.equal(kh.view(torch.int16), k.view(torch.int16))


@pytest.mark.parametrize("static", [False, True])
def test_host_stream_cp_segments(dev, static):
    """A load-balanced context-parallel rank (cp = 2, rank 0: chunks 0 and 3 of 4) held
    on the host, streamed in chunks that cut across its segments: equal to the same
    rows of a rotation of the whole pack."""
    from packed_varlen_rope_gb300 import cp_shards, shard_rows, shard_segments

    w, pack, q, k = _inputs(2)
    T = pack.total_tokens
    cu = torch.from_numpy(pack.cu_seqlens).to(dev)
    ref_q, ref_k = q.to(dev), k.to(dev)
    pr().rope_qk_bwd(ref_q, ref_k, cu, w.theta)
    shards = cp_shards(T, 2, 0)
    rows = torch.tensor(shard_rows(shards))
    assert int(rows.max()) < T
    sq, sk = q[rows].clone().pin_memory(), k[rows].clone().pin_memory()
    ws = None if static else _workspace(dev, 1000, w)
    pr().rope_qk_host(sq, sk, w.theta, ws, cu_seqlens=cu, segments=shard_segments(shards), backward=True,
                      device=dev)
    torch.cuda.current_stream(dev).synchronize()
    assert torch.equal(sq.view(torch.int16), ref_q.cpu()[rows].view(torch.int16))
    assert torch.equal(sk.view(torch.int16), ref_k.cpu()[rows].view(torch.int16))


def test_host_stream_concurrent_threads(dev):
    """Four host threads call rope_qk_host at the same time, each with its own stream,
    workspace and pack, three calls in a row (forward, backward, forward).  The library
    serialises the enqueueing and orders its shared copy streams with events, so every
    thread ends with exactly what the same three calls give on the device path."""
    import threading

    from packed_varlen_rope_gb300 import workloads as wl

    w, pack, q, k = _inputs(3)
    cu = torch.from_numpy(pack.cu_seqlens).to(dev)
    cache = pr().new_cos_sin_cache(max(pack.lengths), w.head_dim, w.theta, device=dev)
    n = 4
    inputs = [(wl.normal_bf16(q.shape, 610 + i), wl.normal_bf16(k.shape, 620 + i)) for i in range(n)]
    refs = []
    for qi, ki in inputs:
        qd, kd = qi.to(dev), ki.to(dev)
        for backward in (False, True, False):
            (pr().rope_qk_bwd if backward else pr().rope_qk_fwd)(qd, kd, cu, w.theta, cos_sin_cache=cache)
        refs.append((qd.cpu(), kd.cpu()))
    torch.cuda.synchronize()
    results, errors = [None] * n, []

    def worker(i):
        try:
            torch.cuda.set_device(dev)
            s = torch.cuda.Stream(device=dev)
            ws = _workspace(dev, 504 + 8 * i, w)                     # a different chunking per thread
            qh, kh = inputs[i][0].clone().pin_memory(), inputs[i][1].clone().pin_memory()
            for backward in (False, True, False):
                pr().rope_qk_host(qh, kh, w.theta, ws, cu_seqlens=cu, backward=backward, cos_sin_cache=cache,
                                  stream=s)
            s.synchronize()
            results[i] = (qh, kh)
        except Exception as e:                                        # reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(n)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(n):
        assert torch.equal(results[i][0].view(torch.int16), refs[i][0].view(torch.int16)), i
        assert torch.equal(results[i][1].view(torch.int16), refs[i][1].view(torch.int16)), i


@pytest.mark.parametrize("case", range(48))
def test_host_paths_random_options_match_oracle(dev, case):
    """Seeded random host-buffer calls against the oracle: random packs (empty samples,
    rows past the pack), head shapes, chunkings (a workspace of 8 to 600 tokens, or the
    library's static array), positions from cu_seqlens with a token offset, a segment
    list or seq_used, or from int32 / int64 ids, forward or backward, in place or into
    separate host outputs, pinned or pageable host memory."""
    rng = np.random.Generator(np.random.PCG64(31000 + case))
    d = int(rng.choice([16, 32, 64, 96, 128]))
    hq = int(rng.integers(1, 9))
    hkv = int(rng.integers(1, hq + 1))
    lengths = rng.integers(0, 300, size=int(rng.integers(1, 9)))
    lengths[rng.random(lengths.size) < 0.2] = 0
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    pack_tokens = int(cu[-1])
    theta = float(rng.choice([1.0e4, 5.0e5, 1.0e6]))
    bwd = bool(rng.integers(0, 2))
    static = bool(rng.integers(0, 2))
    out_of_place = bool(rng.integers(0, 2))
    pinned = bool(rng.integers(0, 3))
    source = str(rng.choice(["cu", "offset", "segments", "seq_used", "ids32", "ids64"]))
    kw = {}
    T = max(1, pack_tokens + int(rng.integers(0, 5)))
    full = oracle.positions(cu, max(pack_tokens, 2 * T + 8))
    if source == "cu":
        pos = full[:T]
        kw["cu_seqlens"] = torch.from_numpy(cu).to(dev)
    elif source == "offset":
        off = int(rng.integers(0, max(1, pack_tokens)))
        T = max(1, int(rng.integers(1, pack_tokens - off + 5)))
        pos = full[off:off + T]
        kw.update(cu_seqlens=torch.from_numpy(cu).to(dev), token_offset=off)
    elif source == "segments":
        cut = int(rng.integers(1, T)) if T > 1 else 0
        starts = [0] + ([cut] if cut else [])
        toks = [int(rng.integers(0, pack_tokens + 4)) for _ in starts]
        ends = starts[1:] + [T]
        tokens = np.concatenate([np.arange(t0, t0 + e - r0) for r0, t0, e in zip(starts, toks, ends)])
        pos = oracle.positions(cu, max(pack_tokens, int(tokens.max()) + 1))[tokens]
        kw.update(cu_seqlens=torch.from_numpy(cu).to(dev), segments=list(zip(starts, toks)))
    elif source == "seq_used":
        used = np.array([int(rng.integers(0, L + 1)) for L in lengths], np.int32)
        pos = full[:T].copy()
        s_of = np.searchsorted(cu[1:], np.arange(T), side="right")
        inside = pos >= 0
        pos[inside & (pos >= used[np.minimum(s_of, lengths.size - 1)])] = -1
        kw.update(cu_seqlens=torch.from_numpy(cu).to(dev), seq_used=torch.from_numpy(used).to(dev))
    else:
        ids = rng.integers(-3, 1 << 24, size=T).astype(np.int64)
        ids[rng.random(T) < 0.05] = (1 << 24) + 5
        if source == "ids64":
            kw["position_ids"] = torch.from_numpy(ids).to(dev)
            pos = np.where((ids >= 0) & (ids < (1 << 24)), ids, -1)
        else:
            ids32 = ids.astype(np.int32)
            kw["position_ids"] = torch.from_numpy(ids32).to(dev)
            pos = np.where((ids32 >= 0) & (ids32 < (1 << 24)), ids32, -1)
    pos = np.asarray(pos, np.int32)

    def bits(shape):
        f = torch.from_numpy(rng.standard_normal(size=shape).astype(np.float32))
        return f.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    qb, kb = bits((T, hq, d)), bits((T, hkv, d))
    qh = torch.from_numpy(qb.view(np.int16).copy()).view(torch.bfloat16)
    kh = torch.from_numpy(kb.view(np.int16).copy()).view(torch.bfloat16)
    if pinned:
        qh, kh = qh.pin_memory(), kh.pin_memory()
    ws = None if static else _workspace_tokens(dev, int(rng.integers(8, 601)), hq, hkv, d)
    if out_of_place:
        qo, ko = torch.full_like(qh, 5.0), torch.full_like(kh, 5.0)
        pr().rope_qk_host(qh, kh, theta, ws, backward=bwd, q_out=qo, k_out=ko, device=dev, **kw)
    else:
        qo, ko = qh, kh
        pr().rope_qk_host(qh, kh, theta, ws, backward=bwd, device=dev, **kw)
    torch.cuda.synchronize()
    what = (case, d, hq, hkv, source, static, out_of_place, bwd, pinned)
    assert np.array_equal(to_bits(qo), oracle.rope_rows(qb, pos, theta, bwd)), what
    assert np.array_equal(to_bits(ko), oracle.rope_rows(kb, pos, theta, bwd)), what
    if out_of_place:
        assert np.array_equal(to_bits(qh), qb) and np.array_equal(to_bits(kh), kb), what


def _workspace_tokens(dev, tokens, hq, hkv, d):
    per_token = (hq + hkv) * d * 2
    return torch.empty(2 * tokens * per_token + 4096, dtype=torch.uint8, device=dev)
