"""The allocation-free entry point rope_qk_host_static (needs a GB300).

It serves callers that may not allocate device memory themselves: it stages the
chunks of a host-resident pack in a device array built into the library instead of a
caller-provided workspace.  Through the C ABI, calls in a row (a forward on one pack,
then a backward on another of a different shape, so each call reuses the array the
previous one left behind) must give what rope_qk_host gives with its own workspace and
what the CPU oracle gives, within the parity bar of the other tests (and bit for bit,
since the rotation kernel reproduces the oracle's arithmetic).  This file is collected
last and also runs alone.
"""
from __future__ import annotations

import ctypes

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


def _desc(pr, q, k, qo, ko, cu, theta, backward, cache):
    T, hq, d = q.shape
    hkv = k.shape[1]
    desc = pr.RopeQKDesc()
    desc.q, desc.q_stride_token, desc.q_stride_head = q.data_ptr(), hq * d, d
    desc.k, desc.k_stride_token, desc.k_stride_head = k.data_ptr(), hkv * d, d
    desc.q_out, desc.q_out_stride_token, desc.q_out_stride_head = qo.data_ptr(), hq * d, d
    desc.k_out, desc.k_out_stride_token, desc.k_out_stride_head = ko.data_ptr(), hkv * d, d
    desc.cu_seqlens, desc.n_seqs = cu.data_ptr(), cu.numel() - 1
    desc.n_q_heads, desc.n_kv_heads, desc.head_dim = hq, hkv, d
    desc.total_tokens, desc.theta, desc.position_scale = T, float(theta), 1.0
    desc.cos_sin_cache = cache.ref()
    desc.backward = 1 if backward else 0
    return desc


def test_static_staging_matches_workspace_entry_and_oracle(dev):
    import packed_varlen_rope_gb300 as pr
    from packed_varlen_rope_gb300 import workloads as wl

    lib = pr.load_library()
    stream = torch.cuda.current_stream(dev)
    # workload 2 (Qwen3-4B shape, 16,384 tokens: 2 chunks of the 32 MiB array) forward,
    # workload 3 (Llama-3-8B shape, packed) backward, then the other direction of each
    for idx, backward in ((2, False), (3, True), (2, True), (3, False)):
        w = wl.WORKLOADS[idx]
        pack = wl.make_pack(w)
        T = pack.total_tokens
        q = wl.normal_bf16((T, w.n_q_heads, w.head_dim), wl.seed(idx, "q"), device="cpu").pin_memory()
        k = wl.normal_bf16((T, w.n_kv_heads, w.head_dim), wl.seed(idx, "k"), device="cpu").pin_memory()
        cu = torch.from_numpy(pack.cu_seqlens).to(dev)
        cache = pr.new_cos_sin_cache(max(pack.lengths), w.head_dim, w.theta, device=dev)
        q_static, k_static = torch.empty_like(q).pin_memory(), torch.empty_like(k).pin_memory()
        q_ref, k_ref = torch.empty_like(q).pin_memory(), torch.empty_like(k).pin_memory()

        desc = _desc(pr, q, k, q_static, k_static, cu, w.theta, backward, cache)
        st = lib.rope_qk_host_static(ctypes.byref(desc), stream.cuda_stream)
        assert st == 0, pr.rope_strerror(st)
        per_token = (w.n_q_heads + w.n_kv_heads) * w.head_dim * 2
        ws = torch.empty(2 * 1024 * per_token, dtype=torch.uint8, device=dev)
        desc = _desc(pr, q, k, q_ref, k_ref, cu, w.theta, backward, cache)
        st = lib.rope_qk_host(ctypes.byref(desc), ws.data_ptr(), ws.numel(), stream.cuda_stream)
        assert st == 0, pr.rope_strerror(st)
        stream.synchronize()

        for x, got, ref in ((q, q_static, q_ref), (k, k_static, k_ref)):
            s = compare(to_bits(got), to_bits(ref), to_bits(x))
            assert_parity(s, ("static staging vs rope_qk_host", idx, backward))
            assert s["bit_mismatch"] == 0
            want = oracle.rope_packed(to_bits(x), pack.cu_seqlens, w.theta, bwd=backward)
            s = compare(to_bits(got), want, to_bits(x))
            assert_parity(s, ("static staging vs oracle", idx, backward))
            assert s["bit_mismatch"] == 0
        # and the inputs were only read
        assert torch.equal(q.view(torch.int16), wl.normal_bf16(q.shape, wl.seed(idx, "q")).view(torch.int16))


def test_static_staging_rejects_oversized_tokens(dev):
    """A token whose Q and K rows exceed the 32 MiB array is refused with a clear code."""
    import packed_varlen_rope_gb300 as pr

    lib = pr.load_library()
    desc = pr.RopeQKDesc()
    hq, hkv, d = 1 << 16, 1 << 10, 256
    desc.n_q_heads, desc.n_kv_heads, desc.head_dim = hq, hkv, d
    desc.total_tokens, desc.theta, desc.position_scale = 4, 1.0e4, 1.0
    desc.q, desc.q_stride_token, desc.q_stride_head = 0x1000, hq * d, d       # never dereferenced
    desc.k, desc.k_stride_token, desc.k_stride_head = 0x2000, hkv * d, d
    desc.cu_seqlens, desc.n_seqs = 0x3000, 1
    st = lib.rope_qk_host_static(ctypes.byref(desc), None)
    assert st == -10 and "32 MiB" in pr.rope_strerror(st)
