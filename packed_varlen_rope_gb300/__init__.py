"""Packed variable-length QK rotary position embedding (RoPE) for GB300 (sm_103a).

The compute path is librope_qk.so (hand-written CUDA behind a C ABI, declared in
``include/rope_qk.h``); this package only marshals arguments to it.  There is no CPU
or PyTorch fallback: every call raises if the library is missing.

    >>> import torch, packed_varlen_rope_gb300 as pr
    >>> pr.rope_qk_fwd(q, k, cu_seqlens, theta=1e6)          # in place, bf16 [T, H, d]
    >>> pr.rope_qk_bwd(dq, dk, cu_seqlens, theta=1e6)        # transpose rotation
"""
from __future__ import annotations

from ._binding import (  # noqa: F401
    EXPORTS,
    GLU_KINDS,
    LIB_PATH,
    ROPE_CU_DECREASING,
    ROPE_CU_NEGATIVE_START,
    ROPE_CU_NONZERO_START,
    ROPE_CU_PAST_END,
    ROPE_FLAG_POSITION_IDS_INT64,
    ROPE_MAX_SEGMENTS,
    CosSinCache,
    RopeCosSinCacheDesc,
    RopeError,
    RopeQKDesc,
    RopeQKLaunch,
    RopeQKSegment,
    glu_bwd,
    glu_fwd,
    load_library,
    new_cos_sin_cache,
    rope_cos_sin_cache_build,
    rope_cos_sin_eval,
    rope_qk_abi_version,
    rope_qk_apply,
    rope_qk_bwd,
    rope_qk_fwd,
    rope_qk_host,
    rope_qk_inv_freq,
    rope_qk_launch_info,
    rope_qk_positions,
    rope_strerror,
    rope_validate_cu_seqlens,
)
from .shards import cp_shards, shard_rows, shard_segments, ulysses_heads  # noqa: F401


def _autograd_function():
    import torch

    class RopeQK(torch.autograd.Function):
        """Autograd wrapper: forward rotates q and k in place (they are marked dirty);
        backward applies the transpose rotation to the incoming gradients."""

        @staticmethod
        def forward(ctx, q, k, theta, cu_seqlens, position_ids, token_offset, position_scale, cos_sin_cache,
                    segments, seq_used):
            rope_qk_apply(q, k, theta, cu_seqlens=cu_seqlens, position_ids=position_ids,
                          token_offset=token_offset, position_scale=position_scale, cos_sin_cache=cos_sin_cache,
                          segments=segments, seq_used=seq_used)
            ctx.mark_dirty(q, k)
            ctx.save_for_backward(cu_seqlens, position_ids, seq_used)
            ctx.args = (theta, token_offset, position_scale, cos_sin_cache, segments)
            return q, k

        @staticmethod
        def backward(ctx, dq, dk):
            cu_seqlens, position_ids, seq_used = ctx.saved_tensors
            theta, token_offset, position_scale, cache, segments = ctx.args
            dq, dk = dq.contiguous(), dk.contiguous()      # e.g. broadcast (stride 0) gradients
            dq_out = torch.empty(dq.shape, dtype=dq.dtype, device=dq.device)
            dk_out = torch.empty(dk.shape, dtype=dk.dtype, device=dk.device)
            # rows the forward left as they were (pad rows under seq_used) pass their
            # gradient through: out of place, the kernel copies them unchanged
            rope_qk_apply(dq, dk, theta, cu_seqlens=cu_seqlens, position_ids=position_ids, backward=True,
                          q_out=dq_out, k_out=dk_out, token_offset=token_offset,
                          position_scale=position_scale, cos_sin_cache=cache, segments=segments,
                          seq_used=seq_used)
            return dq_out, dk_out, None, None, None, None, None, None, None, None

    return RopeQK


_RopeQK = None


def apply_rope_qk(q, k, cu_seqlens, theta: float, cos_sin_cache=None, position_ids=None, token_offset: int = 0,
                  position_scale: float = 1.0, segments=None, seq_used=None):
    """Differentiable in-place RoPE of packed q [T, Hq, d] and k [T, Hkv, d] (any
    token/head strides).  Positions from ``position_ids`` if given, else from
    ``cu_seqlens`` (row r is token ``token_offset + r``, or as ``segments`` map it);
    with ``seq_used`` (int32 [n_seqs]) only the first seq_used[s] rows of sample s are
    rotated and the rest (a padded batch's pad rows) are left as they are, in the
    forward and in the gradient."""
    global _RopeQK
    if _RopeQK is None:
        _RopeQK = _autograd_function()
    segs = None if segments is None else tuple((int(a), int(b)) for a, b in segments)
    return _RopeQK.apply(q, k, theta, cu_seqlens, position_ids, int(token_offset), float(position_scale),
                         cos_sin_cache, segs, seq_used)


def _glu_function():
    import torch

    class GLU(torch.autograd.Function):
        """Autograd wrapper of the gated MLP activation: forward h = act(e) * g into a new
        tensor (e and g saved); backward (de, dg) from the library's backward kernel."""

        @staticmethod
        def forward(ctx, kind, e, g):
            ctx.kind = kind
            ctx.save_for_backward(e, g)
            return glu_fwd(kind, e, g)

        @staticmethod
        def backward(ctx, dh):
            e, g = ctx.saved_tensors
            de, dg = glu_bwd(ctx.kind, dh.contiguous(), e, g)
            return None, de, dg

    return GLU


_GLU = None


def apply_glu(kind: str, e, g):
    """Differentiable h = act(e) * g for bf16 CUDA [rows, cols] views with contiguous rows
    (e.g. the gate and up halves of one fused projection output): ``kind`` "swiglu"
    (SiLU), "geglu" (GELU, erf form) or "geglu_tanh" (GELU, tanh form)."""
    global _GLU
    if kind not in GLU_KINDS:
        raise ValueError("kind must be one of %s" % sorted(GLU_KINDS))
    if _GLU is None:
        _GLU = _glu_function()
    return _GLU.apply(kind, e, g)


def cache_rows_for(needed: int, current: int) -> int:
    """Rows a growing cos/sin cache is built with: ``current`` if it covers ``needed``,
    else the next power of two >= needed (at least 1024), so that a run of growing packs
    rebuilds it O(log) times."""
    if needed <= current:
        return current
    return max(1024, 1 << (int(needed) - 1).bit_length())


class RotaryEmbedding:
    """The rotation of one attention layout (head_dim, theta, linear position_scale)
    with its cos/sin cache managed per device.

    Positions taken from ``cu_seqlens`` are below ``token_offset + T``, a bound known on
    the host, so the cache is grown to that many rows before the call (no device
    synchronisation); with explicit ``position_ids`` it is grown to ``T`` rows and
    positions beyond it are evaluated on the fly, with the same bits.

        >>> rope = RotaryEmbedding(128, 1e6)
        >>> q, k = rope(q, k, cu_seqlens=cu)          # in place, differentiable
    """

    def __init__(self, head_dim: int, theta: float, position_scale: float = 1.0, use_cache: bool = True):
        """``use_cache=False``: no table at all, cos/sin evaluated in the kernel (the same
        bits; as fast on large packs, a few % slower on small ones, and no memory: the
        table of a 1,048,576-token sequence with head_dim 128 takes 512 MiB)."""
        if head_dim % 16 != 0 or not 16 <= head_dim <= 256:
            raise ValueError("head_dim must be a multiple of 16 in [16, 256]")
        self.head_dim, self.theta, self.position_scale = int(head_dim), float(theta), float(position_scale)
        self.use_cache = bool(use_cache)
        self._caches = {}

    def cache(self, device, rows: int):
        """The cos/sin cache of ``device`` with at least ``rows`` rows (built or grown)."""
        import torch

        device = torch.device(device)
        cur = self._caches.get(device)
        want = cache_rows_for(rows, 0 if cur is None else cur.rows)
        if cur is None or want != cur.rows:
            cur = new_cos_sin_cache(want, self.head_dim, self.theta, device=device,
                                    position_scale=self.position_scale)
            self._caches[device] = cur
        return cur

    def __call__(self, q, k, cu_seqlens=None, position_ids=None, token_offset: int = 0,
                 max_position: int = 0, segments=None, seq_used=None):
        """Rotate q and k in place (differentiable).  ``max_position``: an upper bound on
        the position ids, for ids that exceed the row count (a context-parallel shard
        of a long sequence carrying global ids); without it the cache covers ``T``
        rows and larger ids are evaluated on the fly.  ``segments``: a context-parallel
        rank's (row_start, token_start) list (``shard_segments``).  ``seq_used``: the
        tokens used per sample of a padded batch (pad rows left as they are)."""
        if q.shape[-1] != self.head_dim:
            raise ValueError("q and k must have head_dim %d" % self.head_dim)
        T = q.shape[0]
        if position_ids is not None:
            rows = T
        elif segments is not None:
            segs = list(segments)
            ends = [segs[i + 1][0] if i + 1 < len(segs) else T for i in range(len(segs))]
            rows = max(b + (e - a) for (a, b), e in zip(segs, ends))
        else:
            rows = int(token_offset) + T
        rows = max(rows, int(max_position) + 1 if max_position else 0)
        cache = self.cache(q.device, max(rows, 1)) if self.use_cache else None
        return apply_rope_qk(q, k, cu_seqlens, self.theta, cos_sin_cache=cache, position_ids=position_ids,
                             token_offset=token_offset, position_scale=self.position_scale, segments=segments,
                             seq_used=seq_used)
