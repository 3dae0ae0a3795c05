"""Multi-rank host logic of the benchmark on CPU: 2 gloo ranks, no GPU.

Each rank rotates its own pack (seeds offset by rank); the whole-job value is the
tokens of all ranks over the slowest rank's time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from packed_varlen_rope_gb300 import workloads as wl

    pack = wl.make_pack(wl.WORKLOADS[4], rank=rank)
    ms = [1.5, 2.5][rank]
    worst = bench.max_over_ranks(ms, world)
    value = bench.whole_job_tokens_per_s(world, pack.valid_tokens, worst)
    out[rank] = (pack.cu_seqlens.tolist(), pack.valid_tokens, worst, value)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_gloo_ranks():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    cu0, t0, worst0, v0 = out[0]
    cu1, t1, worst1, v1 = out[1]
    assert cu0 != cu1                                   # independent packs per rank
    assert t0 == t1 == 65536                            # same work per rank (weak scaling)
    assert worst0 == worst1 == 2.5                      # slowest rank's time on every rank
    assert v0 == v1 == pytest.approx(2 * 65536 / 2.5e-3)


def _cp_rank_main(rank, world, port, out):
    """One context-parallel rank: its load-balanced shards of the Llama-3-8B-shape pack
    (7,714 packed tokens, padded to a multiple of 2 * world), rotated by the CPU oracle
    with the global positions the shard plan gives; rank 0 gathers every rank's rows."""
    import numpy as np
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from packed_varlen_rope_gb300 import cp_shards, shard_rows, shard_segments
    from packed_varlen_rope_gb300 import workloads as wl

    oracle.build()
    w = wl.WORKLOADS[3]
    pack = wl.make_pack(w)
    T = pack.total_tokens
    bits = lambda shape, kind: wl.normal_bf16(shape, wl.seed(3, kind)).view(__import__("torch").int16) \
        .numpy().view(np.uint16)                                       # the same pack on every rank
    x = {"q": bits((T, w.n_q_heads, w.head_dim), "q"), "k": bits((T, w.n_kv_heads, w.head_dim), "k")}
    shards = cp_shards(T, world, rank, load_balanced=True)
    rows = np.array(shard_rows(shards))
    # the segments map local rows to the same global tokens
    segs = shard_segments(shards)
    from_segs = np.concatenate([np.arange(tok, tok + ((segs[i + 1][0] if i + 1 < len(segs) else rows.size) - r0))
                                for i, (r0, tok) in enumerate(segs)])
    assert np.array_equal(from_segs, rows)
    pos = oracle.positions(pack.cu_seqlens, max(T, int(rows.max()) + 1))[rows]   # padding rows: -1
    local = {}
    for name, full in x.items():
        xl = np.zeros((rows.size,) + full.shape[1:], np.uint16)
        inside = rows < T
        xl[inside] = full[rows[inside]]
        local[name] = oracle.rope_rows(xl, pos, w.theta, bwd=(name == "k"))
    gathered = [None] * world if rank == 0 else None
    dist.gather_object((rows, local), gathered, dst=0)
    if rank == 0:
        seen = np.zeros(T, np.int32)
        got = {name: np.zeros_like(full) for name, full in x.items()}
        for r_rows, r_local in gathered:
            inside = r_rows < T
            seen[r_rows[inside]] += 1
            for name in got:
                got[name][r_rows[inside]] = r_local[name][inside]
        ok = bool(np.all(seen == 1))
        ok = ok and np.array_equal(got["q"], oracle.rope_packed(x["q"], pack.cu_seqlens, w.theta))
        ok = ok and np.array_equal(got["k"], oracle.rope_packed(x["k"], pack.cu_seqlens, w.theta, bwd=True))
        out["ok"] = ok
        out["padding_rows"] = int(sum((r >= T).sum() for r, _ in gathered))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_cp_shards_across_gloo_ranks_equal_the_whole_pack():
    """Two gloo ranks each rotate their load-balanced context-parallel shards (chunks r
    and 3 - r of 4) with the oracle; gathered in pack order, every token appears once and
    the result equals the oracle's rotation of the whole pack bit for bit."""
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_cp_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out["ok"]
    assert out["padding_rows"] == 2                     # 7,714 tokens padded to 4 chunks of 1,929
