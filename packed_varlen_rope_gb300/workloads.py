"""Seeded synthetic workloads for packed variable-length QK-RoPE.

This module only draws random numbers and lays out packing metadata; it holds none
of the rotation arithmetic, so both the CUDA path and the CPU oracle may take their
inputs from it.

The five workloads follow the shapes the source pages train on (unsloth.ai "3x faster
training with packing": Qwen3-4B/8B/32B and Llama-3-8B fine-tunes on many short rows
with some long ones; TRL "training beyond 1M tokens": one 1M-token sequence).  The
pages' datasets are not available, so seeded length mixtures stand in for them:

* lengths: numpy ``PCG64(1000 + c)``; each sample picks a length range by a
  Bernoulli draw, then an inclusive uniform integer in that range; samples are drawn
  until their sum reaches ``total_tokens`` and the last one is cut to fit;
* values: bf16 from float32 N(0, 1) draws (round to nearest even), torch generators
  seeded ``2000 + c`` (Q), ``3000 + c`` (K), ``4000 + c`` (dQ), ``5000 + c`` (dK);
* sampled check rows for the 1M-token pack: ``PCG64(6000 + c)``.

A rank of a multi-process run adds ``rank * 100_000`` to every seed, so each rank
rotates its own pack.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np

RANK_SEED_STRIDE = 100_000


@dataclass(frozen=True)
class Workload:
    index: int                      # 1-based workload number
    name: str
    total_tokens: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    theta: float
    # Either fixed lengths, or a mixture [(probability, lo, hi), ...] drawn to total_tokens.
    lengths: Optional[Tuple[int, ...]] = None
    mixture: Optional[Tuple[Tuple[float, int, int], ...]] = None
    # Padded-vs-packed workload: n samples of U[lo, hi], padded to n * pad_to.
    padded_samples: Optional[Tuple[int, int, int, int]] = None   # (n, lo, hi, pad_to)
    description: str = ""

    @property
    def half(self) -> int:
        return self.head_dim // 2


WORKLOADS = {
    1: Workload(1, "tiny-pack-4x", 64, 4, 2, 64, 1.0e4, lengths=(5, 17, 33, 9),
                description="4 sequences {5,17,33,9} packed, Q 4 / K 2 heads, d 64, theta 1e4"),
    2: Workload(2, "qwen3-4b-16k", 16_384, 32, 8, 128, 1.0e6,
                mixture=((0.8, 32, 512), (0.2, 2048, 8192)),
                description="Qwen3-4B attention shape, 16,384 tokens, 80% U[32,512] / 20% U[2048,8192]"),
    3: Workload(3, "llama3-8b-8x2048", 8 * 2048, 32, 8, 128, 5.0e5,
                padded_samples=(8, 64, 2048, 2048),
                description="Llama-3-8B shape, 8 samples U[64,2048], padded to 8x2048 and packed"),
    4: Workload(4, "qwen3-32b-64k", 65_536, 64, 8, 128, 1.0e6,
                mixture=((0.5, 16, 256), (0.5, 1024, 4096)),
                description="Qwen3-32B attention shape, 65,536 tokens, 50% U[16,256] / 50% U[1024,4096]"),
    5: Workload(5, "long-1m-int64", 1 << 20, 32, 8, 128, 1.0e6, lengths=(1 << 20,),
                description="one 1,048,576-token sequence, Q 32 / K 8 heads, d 128 (Q numel 2^32)"),
}


def seed(workload: int, kind: str, rank: int = 0) -> int:
    base = {"lengths": 1000, "q": 2000, "k": 3000, "dq": 4000, "dk": 5000, "rows": 6000}[kind]
    return base + workload + RANK_SEED_STRIDE * rank


def draw_lengths(w: Workload, rank: int = 0) -> List[int]:
    """Sample lengths of the packed samples (sum == total_tokens, except padded workloads)."""
    if w.lengths is not None:
        return list(w.lengths)
    rng = np.random.Generator(np.random.PCG64(seed(w.index, "lengths", rank)))
    if w.padded_samples is not None:
        n, lo, hi, _ = w.padded_samples
        return [int(rng.integers(lo, hi + 1)) for _ in range(n)]
    assert w.mixture is not None
    lengths: List[int] = []
    total = 0
    probs = [m[0] for m in w.mixture]
    while total < w.total_tokens:
        u = rng.random()
        acc = 0.0
        pick = len(w.mixture) - 1
        for i, p in enumerate(probs):
            acc += p
            if u < acc:
                pick = i
                break
        _, lo, hi = w.mixture[pick]
        n = int(rng.integers(lo, hi + 1))
        n = min(n, w.total_tokens - total)
        lengths.append(n)
        total += n
    return lengths


def cu_from_lengths(lengths: Sequence[int]) -> np.ndarray:
    """Packing metadata: int32 [n+1] offsets of each sample in the 1-D token stream."""
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    assert cu[-1] < 2**31
    return cu.astype(np.int32)


@dataclass
class Pack:
    workload: Workload
    lengths: List[int]
    cu_seqlens: np.ndarray          # int32 [n+1]
    total_tokens: int
    layout: str                     # "packed" or "padded"
    valid_mask: Optional[np.ndarray] = field(default=None)   # bool [T] for padded layout

    @property
    def n_seqs(self) -> int:
        return len(self.cu_seqlens) - 1

    @property
    def valid_tokens(self) -> int:
        return int(sum(self.lengths))


def make_pack(w: Workload, layout: str = "packed", rank: int = 0) -> Pack:
    lengths = draw_lengths(w, rank)
    if layout == "packed":
        cu = cu_from_lengths(lengths)
        return Pack(w, lengths, cu, int(cu[-1]), "packed")
    assert layout == "padded" and w.padded_samples is not None
    n, _, _, pad_to = w.padded_samples
    cu = cu_from_lengths([pad_to] * n)
    mask = np.zeros(n * pad_to, dtype=bool)
    for b, L in enumerate(lengths):
        mask[b * pad_to: b * pad_to + L] = True
    return Pack(w, lengths, cu, n * pad_to, "padded", valid_mask=mask)


def normal_bf16(shape, seed_value: int, device="cpu", chunk_elems: int = 1 << 28):
    """bf16 tensor of N(0,1) float32 draws rounded to nearest even, drawn in chunks so a
    multi-GB tensor needs no float32 copy of itself."""
    import torch

    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    g = torch.Generator(device=device)
    g.manual_seed(int(seed_value))
    n = flat.numel()
    for start in range(0, n, chunk_elems):
        stop = min(n, start + chunk_elems)
        flat[start:stop].copy_(torch.randn(stop - start, generator=g, device=device,
                                           dtype=torch.float32))
    return out


def sampled_rows(w: Workload, n_random: int = 4096, rank: int = 0) -> np.ndarray:
    """Sorted unique token indices to check on a pack too large for the oracle in full:
    seeded random tokens plus the tokens where Q's flat element offset crosses 2^31
    and the ends of the pack."""
    T = w.total_tokens
    rng = np.random.Generator(np.random.PCG64(seed(w.index, "rows", rank)))
    rand = rng.integers(0, T, size=n_random)
    per_token = w.n_q_heads * w.head_dim
    cross = (1 << 31) // per_token
    fixed = [0, 1, T - 1, cross - 1, cross, cross + 1]
    rows = np.unique(np.concatenate([rand, np.asarray([f for f in fixed if 0 <= f < T])]))
    return rows.astype(np.int64)


@dataclass(frozen=True)
class GluWorkload:
    name: str
    rows: int            # tokens
    cols: int            # MLP intermediate width
    kind: str            # "swiglu", "geglu" or "geglu_tanh"
    description: str = ""


# The MLP of the TRL page's long-context section: 1,048,576 tokens, each widened from
# 2,560 to 9,728 (Qwen3-4B), act_fn = SiLU; and a 64k-token slice of it.
GLU_WORKLOADS = {
    "qwen3-4b-mlp-1m": GluWorkload("qwen3-4b-mlp-1m", 1 << 20, 9728, "swiglu",
                                   "1,048,576 tokens x 9,728 (10.2e9 elements per matrix, int64 offsets)"),
    "qwen3-4b-mlp-64k": GluWorkload("qwen3-4b-mlp-64k", 65_536, 9728, "swiglu",
                                    "65,536 tokens x 9,728"),
    "qwen3-4b-mlp-16k": GluWorkload("qwen3-4b-mlp-16k", 16_384, 9728, "swiglu",
                                    "16,384 tokens x 9,728 (319 MB per matrix; profiling size)"),
}
