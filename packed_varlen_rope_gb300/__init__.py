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
    RopeError,
    RopeQKDesc,
    glu_bwd,
    glu_fwd,
    load_library,
    new_cos_sin_cache,
    rope_cos_sin_cache_build,
    rope_qk_abi_version,
    rope_qk_apply,
    rope_qk_bwd,
    rope_qk_fwd,
    rope_qk_host,
    rope_qk_inv_freq,
    rope_qk_positions,
    rope_strerror,
    rope_validate_cu_seqlens,
)


def _autograd_function():
    import torch

    class RopeQK(torch.autograd.Function):
        """Autograd wrapper: forward rotates q and k in place (they are marked dirty);
        backward applies the transpose rotation to the incoming gradients."""

        @staticmethod
        def forward(ctx, q, k, cu_seqlens, theta, cos_sin_cache):
            rope_qk_fwd(q, k, cu_seqlens, theta, in_place=True, cos_sin_cache=cos_sin_cache)
            ctx.mark_dirty(q, k)
            ctx.save_for_backward(cu_seqlens, cos_sin_cache)
            ctx.theta = theta
            return q, k

        @staticmethod
        def backward(ctx, dq, dk):
            cu_seqlens, cache = ctx.saved_tensors
            dq = dq.contiguous()
            dk = dk.contiguous()
            dq_out = torch.empty_like(dq)
            dk_out = torch.empty_like(dk)
            rope_qk_bwd(dq, dk, cu_seqlens, ctx.theta, in_place=False, q_out=dq_out, k_out=dk_out,
                        cos_sin_cache=cache)
            return dq_out, dk_out, None, None, None

    return RopeQK


_RopeQK = None


def apply_rope_qk(q, k, cu_seqlens, theta: float, cos_sin_cache=None):
    """Differentiable in-place RoPE of packed q [T, Hq, d] and k [T, Hkv, d]."""
    global _RopeQK
    if _RopeQK is None:
        _RopeQK = _autograd_function()
    return _RopeQK.apply(q, k, cu_seqlens, theta, cos_sin_cache)
