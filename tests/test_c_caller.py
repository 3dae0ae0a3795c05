"""A C program calling librope_qk.so (tests/c_caller/rope_c_caller.c), compiled with
gcc against include/rope_qk.h and linked with -lrope_qk -lcudart.

On CPU: it compiles and links.  On a GB300 (-m gpu): it runs the tiny pack (4 samples
{5, 17, 33, 9}, Q 4 / K 2 heads, d 64, theta 1e4) through cudaMalloc'd buffers, the
forward rotation with a cos/sin cache and the backward without one, and its outputs
equal the CPU oracle bit for bit."""
from __future__ import annotations

import glob
import os
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SOURCE = os.path.join(ROOT, "tests", "c_caller", "rope_c_caller.c")


def _cuda_home():
    from packed_varlen_rope_gb300 import build

    return os.path.dirname(os.path.dirname(os.path.realpath(build.nvcc())))


def _cuda_libdir(home):
    for cand in [os.path.join(home, "lib64")] + sorted(glob.glob(os.path.join(home, "targets", "*", "lib"))):
        if os.path.exists(os.path.join(cand, "libcudart.so")):
            return cand
    pytest.skip("no libcudart.so next to nvcc")


def build_caller(out_dir) -> str:
    from packed_varlen_rope_gb300 import build

    lib = build.build()
    home = _cuda_home()
    libdir = _cuda_libdir(home)
    exe = os.path.join(str(out_dir), "rope_c_caller")
    pkg = os.path.dirname(lib)
    subprocess.check_call(["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror",
                           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(home, "include"),
                           SOURCE, "-o", exe, "-L", pkg, "-lrope_qk", "-L", libdir, "-lcudart",
                           "-Wl,-rpath," + pkg + ":" + libdir])
    return exe


def test_c_caller_compiles_and_links(tmp_path):
    exe = build_caller(tmp_path)
    assert os.access(exe, os.X_OK)


@pytest.mark.gpu
def test_c_caller_matches_oracle(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from packed_varlen_rope_gb300 import workloads as wl

    oracle.build()
    exe = build_caller(tmp_path)
    w = wl.WORKLOADS[1]
    pack = wl.make_pack(w)
    T = pack.total_tokens
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    q = bits(wl.normal_bf16((T, w.n_q_heads, w.head_dim), wl.seed(1, "q")))
    k = bits(wl.normal_bf16((T, w.n_kv_heads, w.head_dim), wl.seed(1, "k")))
    inp, outp = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(inp, "wb") as f:
        f.write(np.array([T, w.n_q_heads, w.n_kv_heads, w.head_dim, pack.n_seqs], "<i4").tobytes())
        f.write(np.array([w.theta], "<f8").tobytes())
        f.write(pack.cu_seqlens.astype("<i4").tobytes())
        f.write(q.astype("<u2").tobytes())
        f.write(k.astype("<u2").tobytes())
    run = subprocess.run([exe, str(inp), str(outp)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    assert run.stdout.strip().endswith("ok"), run.stdout
    out = np.fromfile(outp, dtype="<u2")
    nq, nk = q.size, k.size
    assert out.size == 2 * (nq + nk)
    fq, fk = out[:nq].reshape(q.shape), out[nq:nq + nk].reshape(k.shape)
    bq, bk = out[nq + nk:2 * nq + nk].reshape(q.shape), out[2 * nq + nk:].reshape(k.shape)
    rq = oracle.rope_packed(q, pack.cu_seqlens, w.theta)
    rk = oracle.rope_packed(k, pack.cu_seqlens, w.theta)
    assert np.array_equal(fq, rq) and np.array_equal(fk, rk)
    assert np.array_equal(bq, oracle.rope_packed(rq, pack.cu_seqlens, w.theta, bwd=True))
    assert np.array_equal(bk, oracle.rope_packed(rk, pack.cu_seqlens, w.theta, bwd=True))
