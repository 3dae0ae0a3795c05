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
