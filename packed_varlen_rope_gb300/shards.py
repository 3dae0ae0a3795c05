"""Context-parallel shard plan of a packed sequence (host logic only, no GPU).

The TRL page "training beyond 1M tokens" (context-parallel section) splits a long
sequence across ``cp_size`` ranks.  Two layouts:

* contiguous: the sequence, padded to a multiple of ``cp_size``, is cut into
  ``cp_size`` equal chunks and rank r holds chunk r;
* load-balanced (the page's ``2 * cp_size`` chunking for causal attention): padded to
  a multiple of ``2 * cp_size`` and cut into ``2 * cp_size`` equal chunks, rank r holds
  chunks r and ``2 * cp_size - 1 - r``, so every rank gets one early and one late chunk.

A rank's local Q and K rows are its chunks one after the other.  The rotation needs
only each row's global token index in the pack's ``cu_seqlens`` stream: the shard's
``(row_start, token_start)`` segments give it, and one call of ``rope_qk_apply`` with
``segments=`` rotates every shard of the rank.  Rows whose token index is at or past
the pack's end (the padding) lie outside every sample and are left as they are.
"""
from __future__ import annotations

from typing import List, Tuple


def cp_shards(total_tokens: int, cp_size: int, rank: int, load_balanced: bool = True) -> List[Tuple[int, int]]:
    """The chunks of the pack rank ``rank`` holds, in local row order, as
    ``(token_start, n_rows)`` pairs (the padding to equal chunks included)."""
    T, cp, r = int(total_tokens), int(cp_size), int(rank)
    if T < 0 or cp < 1 or not 0 <= r < cp:
        raise ValueError("need total_tokens >= 0, cp_size >= 1 and 0 <= rank < cp_size")
    if not load_balanced:
        chunk = -(-T // cp)
        return [(r * chunk, chunk)]
    chunk = -(-T // (2 * cp))
    return [(r * chunk, chunk), ((2 * cp - 1 - r) * chunk, chunk)]


def shard_segments(shards) -> List[Tuple[int, int]]:
    """``(row_start, token_start)`` segments of a rank's local rows (``rope_qk_apply``'s
    ``segments=``); empty chunks are dropped."""
    segs, row = [], 0
    for token_start, n in shards:
        if n > 0:
            segs.append((row, int(token_start)))
            row += int(n)
    return segs


def shard_rows(shards) -> List[int]:
    """Global token index of every local row of a rank, in order."""
    out: List[int] = []
    for token_start, n in shards:
        out.extend(range(int(token_start), int(token_start) + int(n)))
    return out


def ulysses_heads(n_q_heads: int, n_kv_heads: int, sp_size: int, rank: int):
    """Head shard of a rank under Ulysses sequence parallelism (the DeepSpeed
    alternative the TRL page names next to context parallelism): after the all-to-all
    each rank holds every token of its attention heads.  Returns ((q_lo, q_hi),
    (kv_lo, kv_hi)), half-open head ranges of Q and K.  Q heads are split evenly; K/V
    heads too when there are enough, else each rank keeps the one K/V head its Q heads
    share (grouped-query attention).  The rotation needs no exchange: the rank rotates
    q[:, q_lo:q_hi] and k[:, kv_lo:kv_hi] (strided views) with the pack's cu_seqlens."""
    hq, hkv, sp, r = int(n_q_heads), int(n_kv_heads), int(sp_size), int(rank)
    if hq < 1 or hkv < 1 or sp < 1 or not 0 <= r < sp or hq % sp or hq % hkv:
        raise ValueError("need sp_size | n_q_heads, n_kv_heads | n_q_heads and 0 <= rank < sp_size")
    q_per = hq // sp
    if hkv % sp == 0:
        kv_per = hkv // sp
        return (r * q_per, (r + 1) * q_per), (r * kv_per, (r + 1) * kv_per)
    if sp % hkv:
        raise ValueError("n_kv_heads must divide sp_size or be a multiple of it")
    group = hq // hkv                         # Q heads per K/V head
    kv = (r * q_per) // group
    if ((r + 1) * q_per - 1) // group != kv:
        raise ValueError("a rank's Q heads would span several K/V heads")
    return (r * q_per, (r + 1) * q_per), (kv, kv + 1)
