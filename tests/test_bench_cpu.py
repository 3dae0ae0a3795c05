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


def test_profile_traffic_only_for_the_current_kernel(tmp_path, monkeypatch):
    """The bench reports ncu traffic only from a summary taken on the kernel source as
    it is now (its recorded hash equals the current one); any other summary, or none,
    gives null."""
    summary = tmp_path / "rope_qk_tile_kernel_%s.md"
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(summary))
    (tmp_path / "rope_qk_tile_kernel_now.md").write_text(
        "kernel_source_sha256: %s\ntraffic_bytes_per_launch: 123\n" % bench.kernel_source_hash())
    (tmp_path / "rope_qk_tile_kernel_old.md").write_text(
        "kernel_source_sha256: %s\ntraffic_bytes_per_launch: 456\n" % ("0" * 64))
    assert bench.profiled_traffic("now") == 123
    assert bench.profiled_traffic("old") is None
    assert bench.profiled_traffic("missing") is None


def test_committed_profile_is_current():
    """The workload-4 ncu summary in profiles/ was taken on the kernel as it is now, so
    the bench line carries its DRAM traffic."""
    assert bench.profiled_traffic("qwen3-32b-64k") == 2357833500


def test_whole_job_value_is_weak_scaling():
    assert bench.whole_job_tokens_per_s(4, 65536, 1.0) == 4 * 65536 / 1e-3


def test_cp_value_is_strong_scaling():
    """Context parallelism splits one pack: the whole pack's tokens over the slowest
    rank's time; an emulated rank on one GPU counts its own tokens."""
    assert bench.cp_tokens_per_s(2, 65536, 32768, 0.5) == 65536 / 0.5e-3
    assert bench.cp_tokens_per_s(1, 65536, 32768, 0.5) == 32768 / 0.5e-3


def test_buffer_sets_keep_small_packs_out_of_l2():
    """A step whose tensors touch less than 4 x L2 cycles through copies until one cycle
    does (capped); the workload-4 step needs no copy, and the config says which."""
    assert bench.buffer_sets(2_415_919_104) == 1
    assert bench.buffer_sets(335_544_320) == 2                     # workload 2
    assert bench.buffer_sets(157_982_720) == 4                     # workload 3 packed
    assert bench.buffer_sets(78_991_360) == 7                      # a cp = 2 rank of workload 3
    for b in (1, 98_304, 10**6, 78_991_360, 157_982_720, 335_544_320):
        n = bench.buffer_sets(b)
        assert 1 <= n <= bench.MAX_BUFFER_SETS
        assert n * b >= 4 * bench.L2_BYTES or n == bench.MAX_BUFFER_SETS
        assert n == 1 or (n - 1) * b < 4 * bench.L2_BYTES         # no more copies than needed
    assert bench.buffer_sets(98_304) == bench.MAX_BUFFER_SETS      # the tiny pack: capped
    assert "> 4 x 129 MB L2" in bench.l2_note(2_415_919_104, 1)
    assert "7 copies" in bench.l2_note(78_991_360, 7) and ">= 4 x" in bench.l2_note(78_991_360, 7)
    assert "< 4 x" in bench.l2_note(98_304, bench.MAX_BUFFER_SETS)


def test_all_core_oracle_timing_runs_every_range():
    """The all-core CPU figure splits the token sample into one range per core and
    rotates all of it (tiny workload, short repeat window)."""
    import oracle
    from packed_varlen_rope_gb300 import workloads as wl

    oracle.build()
    w = wl.WORKLOADS[1]
    pack = wl.make_pack(w)
    rng = np.random.Generator(np.random.PCG64(0))
    q, k, dq, dk = (rng.integers(0, 1 << 16, size=(pack.total_tokens, h, w.head_dim), dtype=np.uint16) & 0x3FFF
                    for h in (w.n_q_heads, w.n_kv_heads, w.n_q_heads, w.n_kv_heads))
    pos = oracle.positions(pack.cu_seqlens, pack.total_tokens)
    r = bench.cpu_all_cores(w, pos, q, k, dq, dk, seconds=0.05)
    assert r["cores"] >= 1 and r["value"] > 0 and r["kind"] == "oracle"
    assert "%d token ranges" % r["cores"] in r["sample"]


def test_padding_waste_algebra():
    """The padded Llama-3-8B batch: valid fraction = sum of the sample lengths over
    8 x 2048 rows; a pack wastes nothing."""
    from packed_varlen_rope_gb300 import workloads as wl

    w = wl.WORKLOADS[3]
    padded, packed = wl.make_pack(w, "padded"), wl.make_pack(w, "packed")
    assert padded.lengths == packed.lengths and padded.total_tokens == 8 * 2048
    assert bench.valid_fraction(padded) == sum(padded.lengths) / (8 * 2048)
    assert int(padded.valid_mask.sum()) == sum(padded.lengths) == packed.total_tokens
    assert bench.valid_fraction(packed) == 1.0
    assert 0.4 < bench.valid_fraction(padded) < 0.6          # U[64, 2048] samples: about half wasted


def test_clock_summary_keeps_the_timed_window():
    """The clock record keeps the samples inside the timed region (median SM clock,
    throttle reasons seen there); with fewer than 3 there it widens to warm-up + timed."""
    c = bench.ClockSampler(0)
    c.thread = object()                                  # rows as the NVML thread records them
    off = ["Not Active"] * 4
    c.rows = [(0.5, 1500.0, 2070.0, off), (1.0, 2070.0, 2070.0, off), (1.001, 2070.0, 2070.0, off),
              (1.002, 2040.0, 2070.0, ["Not Active", "Not Active", "Not Active", "Active"]),
              (1.003, 2070.0, 2070.0, off), (2.0, 1000.0, 2070.0, ["Active"] + off[1:])]
    s = c.summary(0.9, 1.01)
    assert s["window"] == "timed" and s["samples"] == 4 and s["sm_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["sm_max_mhz"] == 2070.0
    s = c.summary(1.5, 1.6)                              # no sample inside: warm-up + timed
    assert s["window"] == "warmup+timed" and s["samples"] == 5


def test_reference_arm_line():
    """bench.py --impl reference times the CPU oracle on the host and prints one JSON
    line with the contract's keys, its own cpu_baseline and an e2e object that moves no
    bytes between host and device."""
    import json
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload", "1",
                        "--steps", "3", "--warmup", "1", "--reference-seconds", "1"],
                       cwd=root, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["steps"] == 3 and d["warmup"] == 1 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "tiny-pack-4x"
    # the config is the one our arm prints for the same arguments (same keys, same values)
    assert set(d["config"]) == {"workload", "total_tokens", "valid_tokens", "n_seqs", "max_seq_len", "n_q_heads",
                                "n_kv_heads", "head_dim", "theta", "layout", "valid_fraction", "parallelism",
                                "l2", "cp_shards", "cos_sin"}
    assert d["config"]["parallelism"] == "dp1 (independent packs)" and d["config"]["cp_shards"] is None
    assert 1 <= d["reference_tokens_per_step"] <= 4096
