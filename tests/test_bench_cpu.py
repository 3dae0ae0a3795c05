"""Host-side helpers of bench.py (no GPU)."""
import numpy as np

import bench


def test_parity_block_counts_bf16_units():
    a = np.array([[0x3F80, 0x3F81, 0x8001, 0x0000]], dtype=np.uint16)
    b = np.array([[0x3F80, 0x3F80, 0x0001, 0x8000]], dtype=np.uint16)
    p = bench.parity_block([a], [b], [a])
    # one unit apart, two units across zero (-tiny to +tiny), and +0 vs -0 differ in bits only
    assert p["elements"] == 4 and p["bit_mismatch"] == 3 and p["max_bf16_ulp"] == 2


def test_kernel_hash_ignores_comments_and_spacing():
    code = "int f(int x) {\n  // comment\n  return x + 1; /* block */\n}\n"
    same = "int f(int x) { return x + 1; }"
    assert bench._code_only(code) == bench._code_only(same)
    assert bench._code_only(code) != bench._code_only(same.replace("+ 1", "+ 2"))


def test_committed_profile_matches_kernel():
    """The traffic figure in profiles/ was taken on the kernel as it is now."""
    assert bench.profiled_traffic() is not None


def test_whole_job_value_is_weak_scaling():
    assert bench.whole_job_tokens_per_s(4, 65536, 1.0) == 4 * 65536 / 1e-3
