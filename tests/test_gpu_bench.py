"""bench.py's measurement modes on small workloads (needs a GB300): each prints one
JSON line with the keys its consumers read, and the self-checking forms mode finds
every input form's result equal to the contiguous path's (or to the oracle)."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, timeout=600):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def test_rope_forms_on_qwen3_4b_16k():
    d = _bench("--path", "rope-forms", "--workload", "2")
    assert d["workload"] == "qwen3-4b-16k" and len(d["forms"]) == 11
    for name, f in d["forms"].items():
        assert f["us"] > 0 and f["gbs"] > 0, name
        assert f["check"].startswith("bit-identical") or f["check"].endswith(" 0 differ"), (name, f["check"])


def test_glu_bench_line_on_16k_slice():
    d = _bench("--path", "glu", "--glu-workload", "qwen3-4b-mlp-16k", "--glu-kind", "geglu",
               "--steps", "5", "--warmup", "3")
    k = d["roofline"]["kernels"]
    assert d["config"]["kind"] == "geglu" and d["gpu_launches"] == 10
    assert k["glu_fwd"]["algorithmic_bytes_per_launch"] == 6 * 16384 * 9728
    assert k["glu_bwd"]["algorithmic_bytes_per_launch"] == 10 * 16384 * 9728
    assert 0 < k["glu_fwd"]["frac"] < 2 and 0 < k["glu_bwd"]["frac"] < 2


def test_rope_bench_line_small():
    d = _bench("--workload", "2", "--steps", "20", "--warmup", "3", "--e2e-steps", "2", "--cpu-seconds", "1")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "roofline",
                "cpu_baseline", "cpu_baseline_all_cores", "e2e", "clocks", "gpu_launches", "parity"):
        assert key in d, key
    assert d["parity"]["bit_mismatch"] == 0 and d["gpu_launches"] == 40
    assert d["roofline"]["kernel"] == "rope_qk_tile_kernel<128,false,3>"    # 16,384 1-token tiles, one batch of 3
    assert d["roofline"]["grid"]["ctas"] * d["roofline"]["grid"]["tile_tokens"] >= 16384
    assert d["e2e"]["h2d_bytes_per_step"] == d["e2e"]["d2h_bytes_per_step"] > 0
    assert d["size_matched_copy"]["bytes"] == d["roofline"]["algorithmic_bytes_per_launch"]
    assert d["size_matched_copy"]["gbs"] > 0 and "2 copies" in d["config"]["l2"]
    ref = _bench("--impl", "reference", "--workload", "2", "--steps", "3", "--warmup", "1",
                 "--reference-seconds", "1")
    assert ref["config"] == d["config"]                # both arms describe one workload


@pytest.mark.parametrize("layout", ["padded", "padded-seq-used"])
def test_rope_bench_padded_layouts(layout):
    """The padded Llama-3-8B batch through the bench: every row rotated, or the pad rows
    skipped with seq_used; the oracle parity block and the valid fraction are reported."""
    d = _bench("--workload", "3", "--layout", layout, "--steps", "20", "--warmup", "3", "--e2e-steps", "2",
               "--cpu-seconds", "1")
    assert d["parity"]["bit_mismatch"] == 0 and 0.4 < d["config"]["valid_fraction"] < 0.6
    rows = 16384 if layout == "padded" else d["config"]["valid_tokens"]
    assert d["roofline"]["algorithmic_bytes_per_launch"] == 4 * 40 * 128 * rows


def test_rope_bench_cp_rank():
    """A load-balanced context-parallel rank (cp = 2, rank 1) through the bench: its two
    chunks of the Qwen3-4B-shape pack rotated through the segment list, fwd + bwd back to
    back; the oracle parity block covers the rank's rows, and the value counts its tokens."""
    d = _bench("--workload", "2", "--cp-size", "2", "--cp-rank", "1", "--steps", "20", "--warmup", "3",
               "--e2e-steps", "2", "--cpu-seconds", "1")
    assert d["scaling"] == "strong" and d["config"]["parallelism"].startswith("cp2 (rank 1")
    assert d["config"]["cp_shards"]["rank_tokens"] == 8192
    assert d["config"]["cp_shards"]["segments"] == [[0, 4096], [4096, 8192]]
    assert d["parity"]["bit_mismatch"] == 0 and d["parity"]["elements"] > 0
    assert d["roofline"]["algorithmic_bytes_per_launch"] == 4 * 40 * 128 * 8192
    assert abs(d["value"] - 8192 / (d["ms_per_step"] / 1e3)) < 1e-6 * d["value"]
    ref = _bench("--impl", "reference", "--workload", "2", "--cp-size", "2", "--cp-rank", "1", "--steps", "3",
                 "--warmup", "1", "--reference-seconds", "1")
    assert ref["config"] == d["config"]


def test_rope_head_shapes():
    """Other head shapes (head_dim 64, 80 -- the generic instance --, 96, 128, 256; GQA and
    MHA head counts) through the bench: every sampled row equals the oracle and every
    launch names the instance the library dispatched."""
    d = _bench("--path", "rope-shapes", "--steps", "20", "--warmup", "3", timeout=900)
    assert len(d["shapes"]) == 8
    for name, s in d["shapes"].items():
        assert s["check"].endswith(" 0 differ"), (name, s["check"])
        assert 0 < s["frac"] < 2, name
        dim = int(name.split("/")[2])
        want = dim if dim in (64, 96, 128, 256) else 0
        unroll = 4 if want and s["tokens"] // s["tile_tokens"] >= 32768 else 2   # wide 32-bit launches, a cache
        assert s["kernel"] == "rope_qk_tile_kernel<%d,false,%d>" % (want, unroll), (name, s["kernel"])
