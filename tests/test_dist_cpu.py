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
