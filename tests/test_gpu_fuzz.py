"""Seeded random combinations of the rotation's options against the oracle (needs a
GB300): pack lengths with empty samples, head counts and head_dim, contiguous / fused
QKV / head-major views, in place or out of place, forward or backward, linear rescale,
and positions from cu_seqlens (with a shard offset, a segment list, or seq_used) or
from int32 / int64 position ids with out-of-range values.  Every case must equal the oracle
bit for bit; rows without a position stay unchanged (copied when out of place)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from parity_util import from_bits, to_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
N_CASES = 400


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from packed_varlen_rope_gb300 import build

    build.build()
    oracle.build()
    return torch.device("cuda:0")


def _bits(rng, shape, scale=1.0):
    f = torch.from_numpy((rng.standard_normal(size=shape) * scale).astype(np.float32))
    return f.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _views(buf_kind, T, hq, hkv, d, dev):
    """q and k views of the requested layout over fresh device memory."""
    if buf_kind == "contiguous":
        return (torch.empty((T, hq, d), dtype=torch.bfloat16, device=dev),
                torch.empty((T, hkv, d), dtype=torch.bfloat16, device=dev), None)
    if buf_kind == "fused":
        buf = torch.full((T, hq + 2 * hkv, d), 2.5, dtype=torch.bfloat16, device=dev)
        return buf[:, :hq], buf[:, hq:hq + hkv], buf
    qh = torch.empty((hq, T, d), dtype=torch.bfloat16, device=dev)
    kh = torch.empty((hkv, T, d), dtype=torch.bfloat16, device=dev)
    return qh.transpose(0, 1), kh.transpose(0, 1), None


@pytest.mark.parametrize("case", range(N_CASES))
def test_random_options_match_oracle(dev, case):
    import packed_varlen_rope_gb300 as pr

    rng = np.random.Generator(np.random.PCG64(9000 + case))
    d = int(rng.integers(1, 17)) * 16
    hq = int(rng.integers(1, 9))
    hkv = int(rng.integers(1, hq + 1))
    n_seqs = int(rng.integers(1, 9))
    lengths = rng.integers(0, 200, size=n_seqs)
    lengths[rng.random(n_seqs) < 0.2] = 0                                 # empty samples
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    pack_tokens = int(cu[-1])
    theta = float(rng.choice([1.0e4, 5.0e5, 1.0e6]))
    scale = float(rng.choice([1.0, 1.0, 4.0, 2.5]))
    bwd = bool(rng.integers(0, 2))
    in_place = bool(rng.integers(0, 2))
    layout = str(rng.choice(["contiguous", "fused", "head_major"]))
    source = str(rng.choice(["cu", "cu_offset", "cu_seq_used", "cu_segments", "ids32", "ids64"]))

    # rows of this call and their expected positions (-1: row left as it is)
    if source in ("cu", "cu_seq_used"):
        offset, T = 0, pack_tokens + int(rng.integers(0, 5))          # a few rows past the pack
    elif source == "cu_offset":
        offset = int(rng.integers(0, max(1, pack_tokens)))
        T = int(rng.integers(1, max(2, pack_tokens - offset + 4)))
    elif source == "cu_segments":
        offset, T = 0, int(rng.integers(1, max(2, pack_tokens + 4)))
    else:
        offset, T = 0, int(rng.integers(1, 400))
    T = max(T, 1)
    kw = {}
    if source == "cu_segments":
        # rows cut into 1 to 4 segments, each mapped to its own run of tokens (anywhere in
        # the pack, a few past its end)
        n_seg = int(rng.integers(1, min(4, T) + 1))
        starts = np.sort(rng.choice(np.arange(1, T), size=n_seg - 1, replace=False)) if n_seg > 1 else []
        row_starts = [0] + [int(x) for x in starts]
        token_starts = [int(rng.integers(0, pack_tokens + 4)) for _ in row_starts]
        ends = row_starts[1:] + [T]
        tokens = np.concatenate([np.arange(t0, t0 + (e - r0)) for r0, t0, e in zip(row_starts, token_starts, ends)])
        full = oracle.positions(cu, max(pack_tokens, int(tokens.max()) + 1))
        pos = full[tokens].astype(np.int32)
        kw = {"cu_seqlens": torch.from_numpy(cu).to(dev), "segments": list(zip(row_starts, token_starts))}
    elif source.startswith("cu"):
        full = oracle.positions(cu, max(pack_tokens, offset + T))
        pos = full[offset:offset + T].astype(np.int32)
        kw = {"cu_seqlens": torch.from_numpy(cu).to(dev), "token_offset": offset}
        if source == "cu_seq_used":
            used = np.array([int(rng.integers(0, L + 1)) for L in lengths], np.int32)
            starts = cu[:-1]
            g = np.arange(offset, offset + T)
            s = np.searchsorted(cu[1:], g, side="right")                # sample of each row (if inside)
            inside = pos >= 0
            pos = np.where(inside & (pos < used[np.minimum(s, n_seqs - 1)]), pos, -1).astype(np.int32)
            assert np.all(starts[np.minimum(s, n_seqs - 1)][inside] <= g[inside])
            kw["seq_used"] = torch.from_numpy(used).to(dev)
    else:
        ids = rng.integers(-5, 1 << 24, size=T).astype(np.int64)
        ids[rng.random(T) < 0.05] = (1 << 24) + 3
        if source == "ids64":
            ids[rng.random(T) < 0.05] = (1 << 40) + 7
            kw = {"position_ids": torch.from_numpy(ids).to(dev)}
            pos = np.where((ids >= 0) & (ids < (1 << 24)), ids, -1).astype(np.int32)
        else:
            ids32 = ids.astype(np.int32)
            kw = {"position_ids": torch.from_numpy(ids32).to(dev)}
            pos = np.where((ids32 >= 0) & (ids32 < (1 << 24)), ids32, -1).astype(np.int32)

    vscale = float(rng.choice([1.0, 1.0, 1e-35, 1e35]))              # subnormal products / overflow
    qb, kb = _bits(rng, (T, hq, d), vscale), _bits(rng, (T, hkv, d), vscale)
    q, k, fused = _views(layout, T, hq, hkv, d, dev)
    q.copy_(from_bits(qb, dev))
    k.copy_(from_bits(kb, dev))
    if in_place:
        pr.rope_qk_apply(q, k, theta, backward=bwd, position_scale=scale, **kw)
        qo, ko = q, k
    else:
        qo = torch.full((T, hq, d), 7.0, dtype=torch.bfloat16, device=dev)
        ko = torch.full((T, hkv, d), 7.0, dtype=torch.bfloat16, device=dev)
        pr.rope_qk_apply(q, k, theta, backward=bwd, position_scale=scale, q_out=qo, k_out=ko, **kw)
    torch.cuda.synchronize()
    what = (case, d, hq, hkv, layout, source, in_place, bwd, scale, vscale)
    assert np.array_equal(to_bits(qo.contiguous()), oracle.rope_rows(qb, pos, theta, bwd, scale)), what
    assert np.array_equal(to_bits(ko.contiguous()), oracle.rope_rows(kb, pos, theta, bwd, scale)), what
    if not in_place:
        assert np.array_equal(to_bits(q.contiguous()), qb) and np.array_equal(to_bits(k.contiguous()), kb), what
    if fused is not None:
        assert torch.all(fused[:, hq + hkv:] == 2.5), what                 # V untouched


@pytest.mark.parametrize("case", range(60))
def test_random_glu_options_match_oracle(dev, case):
    """SwiGLU / GeGLU with random shapes, per-matrix row padding, in-place aliasing and
    value scales from 1e-19 (products near the smallest normal bf16) to 1e15 (every
    element on the binary64 path), within the bar of tests/test_gpu_glu.py."""
    import packed_varlen_rope_gb300 as pr
    from test_gpu_glu import KINDS, _fwd_bwd_check

    rng = np.random.Generator(np.random.PCG64(9500 + case))
    kind = str(rng.choice(KINDS))
    rows = int(rng.integers(1, 300))
    cols = int(rng.integers(1, 65)) * 8
    scale = float(rng.choice([1.0, 3.0, 12.0, 40.0, 1e-19, 1e15]))

    def bits():
        f = torch.from_numpy((rng.standard_normal(size=(rows, cols)) * scale).astype(np.float32))
        return f.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    def mat(b=None):
        pad = int(rng.choice([0, 0, 8, 40]))
        buf = torch.full((rows * (cols + pad),), 6.5, dtype=torch.bfloat16, device=dev)
        t = buf.as_strided((rows, cols), (cols + pad, 1))
        if b is not None:
            t.copy_(from_bits(b, dev))
        return t

    eb, gb, dhb = bits(), bits(), bits()
    e, g, dh = mat(eb), mat(gb), mat(dhb)
    in_place = bool(rng.integers(0, 2))
    h = g if in_place else mat()
    pr.glu_fwd(kind, e, g, h)
    torch.cuda.synchronize()
    h_res = h.clone()
    g.copy_(from_bits(gb, dev))                               # restore g if h overwrote it
    de, dg = (e, g) if in_place else (mat(), mat())
    pr.glu_bwd(kind, dh, e, g, de, dg)
    torch.cuda.synchronize()
    _fwd_bwd_check(kind, eb, gb, dhb, h_res, de.clone(), dg.clone(), (case, kind, rows, cols, scale, in_place))
