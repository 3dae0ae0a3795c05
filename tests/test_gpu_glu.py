"""SwiGLU / GeGLU kernels against the binary64 oracle (needs a GB300).

Bar (derived from the arithmetic: the kernels evaluate in binary32 -- special-function
exponentials and reciprocals and a fitted erfc where results stay normal, the accurate
CUDA functions beyond -- the oracle in binary64, both round once to bf16):

    |gpu - ref| <= ulp_bf16(max(|gpu|, |ref|)) + 2^-18 * M

where M is the magnitude of the computed quantity before rounding (|act(e) g| for h,
|dh act(e)| for dg, |dh g| times the sum of the absolute terms of act'(e) for de), so
that a single rounding flip of bf16 plus a few binary32 units of the terms pass and
nothing else does.  The backward's de crosses zero where act' does; there only the
terms' size bounds the error.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from oracle_pins import bits_to_f64, ulp_bf16
from parity_util import from_bits, to_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
KINDS = ("swiglu", "geglu", "geglu_tanh")


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


def _sig(x):
    return 0.5 * (1.0 + np.tanh(0.5 * x))


def _act_terms(kind, x):
    """(|act(x)|, sum of |terms| of act'(x)) in binary64, for error bounds only."""
    from scipy.special import erfc

    if kind == "swiglu":
        s = _sig(x)
        return np.abs(x * s), s * (1 + np.abs(x) * _sig(-x))
    if kind == "geglu":
        Phi = 0.5 * erfc(-x / np.sqrt(2))
        return np.abs(x * Phi), Phi + np.abs(x) * np.exp(-0.5 * x * x) / np.sqrt(2 * np.pi)
    u = np.sqrt(2 / np.pi) * (x + 0.044715 * x ** 3)
    sp, sm = _sig(2 * u), _sig(-2 * u)
    return np.abs(x * sp), sp + 2 * np.abs(x) * sp * sm * np.sqrt(2 / np.pi) * (1 + 3 * 0.044715 * x * x)


def _check(got_bits, ref_bits, mag, what):
    g, r = bits_to_f64(got_bits), bits_to_f64(ref_bits)
    same_inf = np.isinf(g) & np.isinf(r) & (np.sign(g) == np.sign(r))
    with np.errstate(invalid="ignore", over="ignore"):
        tol = ulp_bf16(np.maximum(np.abs(g), np.abs(r))) + 2.0 ** -18 * mag
        bad = ~((np.abs(g - r) <= tol) | same_inf)
    assert not bad.any(), (what, int(bad.sum()), g[bad][:5], r[bad][:5])
    return int(np.count_nonzero(got_bits != ref_bits))


def _bits(rng, shape, scale=1.0):
    f = torch.from_numpy((rng.standard_normal(size=shape) * scale).astype(np.float32))
    return f.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _fwd_bwd_check(kind, eb, gb, dhb, h, de, dg, what):
    e, g, dh = bits_to_f64(eb), bits_to_f64(gb), bits_to_f64(dhb)
    act_mag, dact_terms = _act_terms(kind, e)
    ref_h = oracle.glu_fwd(kind, eb, gb)
    ref_de, ref_dg = oracle.glu_bwd(kind, dhb, eb, gb)
    flips = 0
    if h is not None:
        flips += _check(to_bits(h), ref_h, act_mag * np.abs(g), (what, "h"))
    if de is not None:
        flips += _check(to_bits(de), ref_de, np.abs(dh * g) * dact_terms, (what, "de"))
        flips += _check(to_bits(dg), ref_dg, np.abs(dh) * act_mag, (what, "dg"))
    return flips


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("rows,cols", [(1, 8), (3, 24), (257, 136), (1000, 9728)])
def test_glu_parity(dev, kind, rows, cols):
    rng = np.random.Generator(np.random.PCG64(rows * 7 + cols))
    eb, gb, dhb = (_bits(rng, (rows, cols), 2.0) for _ in range(3))
    e, g, dh = (from_bits(b, dev) for b in (eb, gb, dhb))
    h = pr().glu_fwd(kind, e, g)
    de, dg = pr().glu_bwd(kind, dh, e, g)
    torch.cuda.synchronize()
    flips = _fwd_bwd_check(kind, eb, gb, dhb, h, de, dg, (kind, rows, cols))
    assert flips <= 3 * rows * cols // 100        # bf16 rounding flips are rare


@pytest.mark.parametrize("kind", KINDS)
def test_glu_fused_gate_up_and_in_place(dev, kind):
    """gate and up as the two halves of one [rows, 2I] projection output; the backward
    writes de over e and dg over g, the forward h over g."""
    rng = np.random.Generator(np.random.PCG64(3))
    rows, inter = 300, 1024
    xb = _bits(rng, (rows, 2 * inter), 1.5)
    dhb = _bits(rng, (rows, inter))
    eb, gb = xb[:, :inter].copy(), xb[:, inter:].copy()
    x = from_bits(xb, dev)
    e, g = x[:, :inter], x[:, inter:]
    h = torch.empty((rows, inter), dtype=torch.bfloat16, device=dev)
    pr().glu_fwd(kind, e, g, h)
    dh = from_bits(dhb, dev)
    pr().glu_bwd(kind, dh, e, g, de=e, dg=g)            # in place
    torch.cuda.synchronize()
    xo = to_bits(x)
    e_res = torch.from_numpy(xo[:, :inter].copy().view(np.int16)).view(torch.bfloat16)
    g_res = torch.from_numpy(xo[:, inter:].copy().view(np.int16)).view(torch.bfloat16)
    _fwd_bwd_check(kind, eb, gb, dhb, h, e_res, g_res, (kind, "fused in place"))
    # forward in place over g
    g2 = from_bits(gb, dev)
    pr().glu_fwd(kind, from_bits(eb, dev), g2, g2)
    torch.cuda.synchronize()
    _fwd_bwd_check(kind, eb, gb, dhb, g2, None, None, (kind, "h over g"))


@pytest.mark.parametrize("kind", KINDS)
def test_glu_autograd_on_fused_projection(dev, kind):
    """apply_glu on the gate and up halves of one [rows, 2I] projection output: h and the
    gradients autograd gives the projection are the oracle's (within the bar), each
    half's gradient landing in its own columns."""
    rng = np.random.Generator(np.random.PCG64(11))
    rows, inter = 257, 1024
    xb = _bits(rng, (rows, 2 * inter), 1.5)
    dhb = _bits(rng, (rows, inter))
    eb, gb = xb[:, :inter].copy(), xb[:, inter:].copy()
    x = from_bits(xb, dev).requires_grad_(True)
    h = pr().apply_glu(kind, x[:, :inter], x[:, inter:])
    h.backward(from_bits(dhb, dev))
    torch.cuda.synchronize()
    grad = to_bits(x.grad)
    de = torch.from_numpy(grad[:, :inter].copy().view(np.int16)).view(torch.bfloat16)
    dg = torch.from_numpy(grad[:, inter:].copy().view(np.int16)).view(torch.bfloat16)
    _fwd_bwd_check(kind, eb, gb, dhb, h, de, dg, (kind, "autograd"))
    with pytest.raises(ValueError):
        pr().apply_glu("relu", x[:, :inter], x[:, inter:])


def test_glu_special_values(dev):
    # includes the far left tails where sigmoid, Phi or sigmoid(2u) are tiny but the
    # products are still normal bf16 numbers (-87.5 ... -95 for SiLU, about -10 for the
    # tanh form, -13 for erf)
    vals = np.array([0.0, -0.0, 1.0, -1.0, 8.0, -8.0, 20.0, -20.0, 88.0, -88.0, 100.0, -100.0, 1e-30, -1e-30,
                     -1.2784645, 3.0e38, -3.0e38, 1e-40, -87.5, -89.0, -95.0, -9.9, -10.1, -10.5, -13.0,
                     -13.5], dtype=np.float32)
    rng = np.random.Generator(np.random.PCG64(4))
    shape = (64, 64)
    eb = torch.from_numpy(rng.choice(vals, size=shape).astype(np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)
    gb, dhb = _bits(rng, shape), _bits(rng, shape)
    for kind in KINDS:
        e, g, dh = (from_bits(b, dev) for b in (eb, gb, dhb))
        h = pr().glu_fwd(kind, e, g)
        de, dg = pr().glu_bwd(kind, dh, e, g)
        torch.cuda.synchronize()
        for t in (h, de, dg):
            assert not torch.isnan(t).any()
        _fwd_bwd_check(kind, eb, gb, dhb, h, de, dg, (kind, "special"))


def test_glu_wide_row_stride(dev):
    """gate, up and h side by side in one buffer whose row stride is 2^30 elements, so
    row 1 starts 2 GiB after row 0 and the row term of every address passes 2^31 bytes;
    the gaps between rows keep their canary values."""
    cols, stride, rows = 64, 1 << 30, 3
    n = (rows - 1) * stride + 3 * cols
    store = torch.full((n,), 6.5, dtype=torch.bfloat16, device=dev)
    view = lambda c: store.as_strided((rows, cols), (stride, 1), c * cols)  # noqa: E731
    rng = np.random.Generator(np.random.PCG64(26))
    eb, gb, dhb = (_bits(rng, (rows, cols), 2.0) for _ in range(3))
    e, g, h = view(0), view(1), view(2)
    e.copy_(from_bits(eb, dev))
    g.copy_(from_bits(gb, dev))
    for kind in KINDS:
        pr().glu_fwd(kind, e, g, h)
        torch.cuda.synchronize()
        _fwd_bwd_check(kind, eb, gb, dhb, h.clone(), None, None, (kind, "wide stride"))
    dh = from_bits(dhb, dev)
    pr().glu_bwd("geglu", dh, e, g, de=e, dg=g)
    torch.cuda.synchronize()
    _fwd_bwd_check("geglu", eb, gb, dhb, None, e.clone(), g.clone(), "wide stride bwd")
    gap = store[3 * cols:stride]
    assert torch.all(gap == 6.5) and torch.all(store[stride + 3 * cols:2 * stride] == 6.5)


@pytest.mark.parametrize("kind", KINDS)
def test_glu_long_1m_by_9728(dev, kind):
    """1,048,576 tokens x 9,728 (the TRL page's MLP width at 1M tokens): every matrix
    spans 10.2e9 elements, so addresses pass 2^32 and 2^33 bytes.  Sampled rows, including
    those around element offset 2^31 and 2^32, against the oracle; canaries after the
    last element survive; the backward runs in place (de over e, dg over g)."""
    from packed_varlen_rope_gb300 import workloads as wl

    rows, cols, guard = 1 << 20, 9728, 4096
    n = rows * cols

    def big(seed):
        store = torch.empty(n + guard, dtype=torch.bfloat16, device=dev)
        store[:n].copy_(wl.normal_bf16((n,), seed, device="cuda"))
        store[n:].fill_(6.5)
        return store, store[:n].view(rows, cols)

    es, e = big(21)
    gs, g = big(22)
    ds, dh = big(23)
    hs, h = big(24)
    rng = np.random.Generator(np.random.PCG64(25))
    pick = np.unique(np.concatenate([rng.integers(0, rows, 64), [0, rows - 1, (1 << 31) // cols,
                                                                 (1 << 32) // cols, (1 << 32) // cols + 1]]))
    pick_dev = torch.from_numpy(pick).to(dev)
    eb, gb, dhb = (to_bits(t[pick_dev]) for t in (e, g, dh))
    pr().glu_fwd(kind, e, g, h)
    pr().glu_bwd(kind, dh, e, g, de=e, dg=g)
    torch.cuda.synchronize()
    _fwd_bwd_check(kind, eb, gb, dhb, h[pick_dev], e[pick_dev], g[pick_dev], (kind, "1M x 9728"))
    for store in (es, gs, ds, hs):
        assert torch.all(store[n:] == 6.5)


@pytest.mark.parametrize("padded", ["e", "g", "h", "dh", "de", "dg"])
def test_glu_one_padded_matrix(dev, padded):
    """Exactly one matrix has a row stride wider than its rows (the others are
    contiguous), so each address term of the padded kernels is exercised on its own;
    the gaps between that matrix's rows keep their canaries."""
    rows, cols, stride = 37, 72, 72 + 24
    rng = np.random.Generator(np.random.PCG64(60 + ["e", "g", "h", "dh", "de", "dg"].index(padded)))
    eb, gb, dhb = (_bits(rng, (rows, cols), 2.0) for _ in range(3))
    store = {}

    def mat(name, bits=None):
        if name != padded:
            t = torch.empty((rows, cols), dtype=torch.bfloat16, device=dev)
        else:
            buf = torch.full((rows * stride,), 6.5, dtype=torch.bfloat16, device=dev)
            store[name] = buf
            t = buf.as_strided((rows, cols), (stride, 1))
        if bits is not None:
            t.copy_(from_bits(bits, dev))
        return t

    for kind in KINDS:
        store.clear()
        e, g, dh = mat("e", eb), mat("g", gb), mat("dh", dhb)
        h, de, dg = mat("h"), mat("de"), mat("dg")
        pr().glu_fwd(kind, e, g, h)
        pr().glu_bwd(kind, dh, e, g, de, dg)
        torch.cuda.synchronize()
        _fwd_bwd_check(kind, eb, gb, dhb, h.clone(), de.clone(), dg.clone(), (kind, padded))
        gaps = store[padded].view(rows, stride)[:, cols:]
        assert torch.all(gaps == 6.5), (kind, padded)
