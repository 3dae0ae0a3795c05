"""The entry points inside a captured CUDA graph (needs a GB300): none of them
synchronises or allocates, and rope_qk_host joins its copy streams to the caller's
stream through events, so a training step that captures them replays them exactly.
One graph holds a forward on (Q, K), a backward on (dQ, dK), the backward of a
context-parallel rank's buffer through a segment list with cos/sin evaluated in the
kernel, a SwiGLU forward and backward and a host-streamed rotation; it is replayed on
fresh inputs copied into the captured buffers and must give what the same calls give
eagerly, bit for bit (the eager results are themselves pinned to the oracle by the
other tests).  The segment list is copied into the kernel's arguments at capture, so
the replay does not depend on the host array."""
from __future__ import annotations

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from packed_varlen_rope_gb300 import build

    build.build()
    return torch.device("cuda:0")


def test_captured_graph_replays_bit_identical(dev):
    import packed_varlen_rope_gb300 as pr
    from packed_varlen_rope_gb300 import workloads as wl

    w = wl.WORKLOADS[2]
    pack = wl.make_pack(w)
    T, hq, hkv, d = pack.total_tokens, w.n_q_heads, w.n_kv_heads, w.head_dim
    cu = torch.from_numpy(pack.cu_seqlens).to(dev)
    cache = pr.new_cos_sin_cache(max(pack.lengths), d, w.theta, device=dev)
    rows, cols = 1024, 2048

    def draw(seed):
        return {"q": wl.normal_bf16((T, hq, d), seed + 1, device=dev),
                "k": wl.normal_bf16((T, hkv, d), seed + 2, device=dev),
                "dq": wl.normal_bf16((T, hq, d), seed + 3, device=dev),
                "dk": wl.normal_bf16((T, hkv, d), seed + 4, device=dev),
                "e": wl.normal_bf16((rows, cols), seed + 5, device=dev),
                "g": wl.normal_bf16((rows, cols), seed + 6, device=dev),
                "dh": wl.normal_bf16((rows, cols), seed + 7, device=dev),
                "hq": wl.normal_bf16((2048, hq, d), seed + 8, device="cpu").pin_memory(),
                "hk": wl.normal_bf16((2048, hkv, d), seed + 9, device="cpu").pin_memory(),
                "cq": wl.normal_bf16((T // 2, hq, d), seed + 10, device=dev),
                "ck": wl.normal_bf16((T // 2, hkv, d), seed + 11, device=dev)}

    per_token = (hq + hkv) * d * 2
    workspace = torch.empty(2 * 512 * per_token, dtype=torch.uint8, device=dev)
    host_cu = torch.tensor([0, 700, 2048], dtype=torch.int32, device=dev)

    segs = pr.shard_segments(pr.cp_shards(T, 2, 1))

    def step(x, out):
        pr.rope_qk_fwd(x["q"], x["k"], cu, w.theta, cos_sin_cache=cache)
        pr.rope_qk_bwd(x["dq"], x["dk"], cu, w.theta, cos_sin_cache=cache)
        pr.rope_qk_apply(x["cq"], x["ck"], w.theta, cu_seqlens=cu, segments=list(segs), backward=True)
        pr.glu_fwd("swiglu", x["e"], x["g"], out["h"])
        pr.glu_bwd("swiglu", x["dh"], x["e"], x["g"], out["de"], out["dg"])
        pr.rope_qk_host(x["hq"], x["hk"], w.theta, workspace, cu_seqlens=host_cu, cos_sin_cache=cache,
                        q_out=out["hq"], k_out=out["hk"])

    def outputs():
        return {"h": torch.empty((rows, cols), dtype=torch.bfloat16, device=dev),
                "de": torch.empty((rows, cols), dtype=torch.bfloat16, device=dev),
                "dg": torch.empty((rows, cols), dtype=torch.bfloat16, device=dev),
                "hq": torch.empty((2048, hq, d), dtype=torch.bfloat16).pin_memory(),
                "hk": torch.empty((2048, hkv, d), dtype=torch.bfloat16).pin_memory()}

    # eager reference on the second draw
    fresh = draw(200)
    eager_in = {n: t.clone() for n, t in fresh.items()}
    eager_out = outputs()
    step(eager_in, eager_out)
    torch.cuda.synchronize()

    # capture on the first draw's buffers (a warm-up on a side stream first, as capture wants)
    static_in, static_out = draw(100), outputs()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step({n: t.clone() for n, t in static_in.items()}, outputs())
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(static_in, static_out)
    for n, t in fresh.items():
        static_in[n].copy_(t)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    for n in ("q", "k", "dq", "dk", "cq", "ck"):
        assert torch.equal(static_in[n], eager_in[n]), n
    for n in ("h", "de", "dg", "hq", "hk"):
        assert torch.equal(static_out[n], eager_out[n]), n
    # a second replay keeps rotating the in-place buffers: equal to two eager steps
    graph.replay()
    step(eager_in, eager_out)
    torch.cuda.synchronize()
    assert torch.equal(static_in["q"], eager_in["q"]) and torch.equal(static_in["dk"], eager_in["dk"])
    assert torch.equal(static_in["cq"], eager_in["cq"]) and torch.equal(static_in["ck"], eager_in["ck"])
