#!/usr/bin/env python
"""Benchmark of fused packed-varlen QK-RoPE, forward + backward, on GB300.

One step = the forward rotation of Q and K and the backward (transpose) rotation of
dQ and dK of one packed batch, in place, through the C ABI of librope_qk.so.  The
default workload is the Qwen3-32B attention shape: 65,536 tokens packed from
50% U[16,256] / 50% U[1024,4096] samples, Q 64 heads, K 8 heads, head_dim 128,
theta 1e6.  The four tensors hold 2.4 GB, far more than the 129 MB L2, so no flush
is needed between steps (a smaller workload's steps cycle through copies of its
tensors, at least 4 x L2 bytes per cycle).  The cos/sin cache is built once before timing, as a model
builds its rotary cache once for all layers and steps.

    python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Prints one JSON line (rank 0).  Under torchrun each rank rotates its own pack (weak
scaling, no collective on the data path); the value is the tokens of all ranks over
the slowest rank's time.  ``--impl reference`` times the CPU oracle on the host cores
instead (bounded samples of the same workload).

Other measurements of the same library:

    --workload N                 another seeded workload (1-5)
    --layout padded|padded-seq-used
                                 the padded batch of workload 3, every row rotated or
                                 the pad rows skipped (value = valid tokens per second)
    --cp-size C [--cp-rank R]    context parallelism over one pack: a rank's load-balanced
                                 chunks rotated through a segment list (torchrun: C ranks,
                                 strong scaling; one GPU: rank R of a group of C)
    --no-cache                   cos/sin evaluated per tile (binary32 double-float, binary64 only
                                 where its rounding is undecided) instead of read from a cache
    --path rope-forms            the forward through every input form (fused QKV,
                                 head-major, out of place, position ids, CP shards, no
                                 cache, rescale), each checked bit for bit
    --path glu                   SwiGLU / GeGLU forward + backward (--glu-workload,
                                 --glu-kind)
    --path rope-shapes           fwd + bwd on other head shapes (head_dim 64, 80, 96, 128,
                                 256; GQA and MHA head counts), ~2.4 GB per launch each,
                                 sampled rows checked against the oracle
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "QK-RoPE fwd+bwd tokens/s and HBM GB/s (% of GB300 peak), packed varlen"
UNIT = "tokens/s"
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 * 10**6          # GB300 L2
MAX_BUFFER_SETS = 64


def buffer_sets(step_bytes: int) -> int:
    """Copies of a step's tensors the timed loop cycles through, so that a launch finds
    none of its inputs in L2: enough that one cycle touches at least 4x the L2 (one set
    when a step alone does), at most MAX_BUFFER_SETS."""
    if step_bytes <= 0:
        return 1
    return int(max(1, min(MAX_BUFFER_SETS, -(-4 * L2_BYTES // step_bytes))))


def size_matched_copy(torch, dev, traffic: int, sets: int, launches: int) -> dict:
    """torch's copy_ moving one launch's bytes (half read, half written) back to back,
    cycling `sets` source/destination pairs as the timed loop cycles its tensors: what
    a plain device copy of the same size reaches, the ramp-up and drain of a short launch
    included.  Reported beside the roofline, whose peak is the long copy's rate."""
    n = max(1, traffic // 4)
    bufs = [(torch.zeros(n, dtype=torch.bfloat16, device=dev), torch.empty(n, dtype=torch.bfloat16, device=dev))
            for _ in range(sets)]
    for i in range(3 * sets):
        bufs[i % sets][1].copy_(bufs[i % sets][0])
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for i in range(launches):
        bufs[i % sets][1].copy_(bufs[i % sets][0])
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / launches
    del bufs
    torch.cuda.empty_cache()
    return {"us_per_copy": us, "gbs": traffic / us / 1e3, "bytes": traffic, "copies": launches}


def l2_note(step_bytes: int, sets: int) -> str:
    """The config's statement of how the timed loop keeps L2 from serving its inputs."""
    if sets == 1:
        return "no flush: Q, K, dQ, dK = %.2f GB per step > 4 x 129 MB L2" % (step_bytes / 1e9)
    cycle = sets * step_bytes
    return ("no flush: steps cycle through %d copies of Q, K, dQ, dK (%.3f GB each, %.2f GB per cycle %s 4 x "
            "129 MB L2)" % (sets, step_bytes / 1e9, cycle / 1e9, ">=" if cycle >= 4 * L2_BYTES else "<"))
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCE = os.path.join(ROOT, "packed_varlen_rope_gb300", "csrc", "rope_qk.cu")
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "rope_qk_tile_kernel_%s.md")   # per workload name


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1, help="GPUs of the run (N > 1: launched under torchrun)")
    ap.add_argument("--steps", type=int, default=2000, help="timed steps (one step: forward + backward)")
    ap.add_argument("--warmup", type=int, default=20, help="untimed steps before them (at least 3 are run)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours",
                    help="ours: the CUDA library; reference: the CPU oracle on the host cores")
    ap.add_argument("--workload", type=int, default=4,
                    help="1 tiny-pack-4x, 2 qwen3-4b-16k, 3 llama3-8b-8x2048, 4 qwen3-32b-64k, 5 long-1m-int64")
    ap.add_argument("--e2e-steps", type=int, default=80, help="timed steps of the host-buffer (e2e) leg")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target seconds of oracle work for the CPU baseline sample")
    ap.add_argument("--reference-seconds", type=float, default=90.0,
                    help="--impl reference: seconds of oracle work over the warm-up and timed steps")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer (e2e) leg")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the CPU oracle baseline and the parity check against it")
    ap.add_argument("--layout", choices=["packed", "padded", "padded-seq-used"], default="packed",
                    help="rope path: the pack as is, or (workloads with padded samples) the padded batch "
                         "with every row rotated, or with the pad rows skipped through seq_used")
    ap.add_argument("--cp-size", type=int, default=1,
                    help="rope path: context parallelism over one pack; each rank holds its load-balanced "
                         "chunks (r and 2*cp-1-r) and rotates them in one launch per pass.  Under torchrun "
                         "the number of ranks; on one GPU, the group size of the rank --cp-rank emulates")
    ap.add_argument("--cp-rank", type=int, default=0, help="rope path, one GPU: the context-parallel rank run")
    ap.add_argument("--no-cache", action="store_true",
                    help="rope path: no cos/sin cache, cos/sin evaluated per tile")
    ap.add_argument("--path", choices=["rope", "glu", "rope-forms", "rope-shapes"], default="rope",
                    help="rope: the QK-RoPE step (default); glu: SwiGLU/GeGLU forward+backward; "
                         "rope-forms: the forward through every input form, each checked; rope-shapes: "
                         "other head shapes")
    ap.add_argument("--glu-workload", default="qwen3-4b-mlp-1m",
                    help="glu path: qwen3-4b-mlp-1m, or its 65,536- and 16,384-token slices")
    ap.add_argument("--glu-kind", choices=["swiglu", "geglu", "geglu_tanh"], default=None,
                    help="activation (default: the workload's)")
    return ap.parse_args()


# ---------------------------------------------------------------- environment

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """C++ source without comments and with whitespace collapsed."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash() -> str:
    """sha256 of the RoPE kernel's device code: rope_qk.cu up to its host-side section,
    then fastdiv.cuh and cos_sin.cuh, comments and whitespace left out.  Host-only edits
    (argument checks, error strings) and comment edits keep it."""
    text = open(KERNEL_SOURCE).read()
    device_part = text.split("// ------------------------------------------------------------------ host side")[0]
    h = hashlib.sha256(_code_only(device_part).encode())
    for header in ("fastdiv.cuh", "cos_sin.cuh"):
        h.update(_code_only(open(os.path.join(os.path.dirname(KERNEL_SOURCE), header)).read()).encode())
    return h.hexdigest()


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary of this workload, if there is
    one and it was taken on the current kernel source; else None."""
    try:
        text = open(PROFILE_SUMMARY % workload).read()
    except OSError:
        return None
    h = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", text)
    t = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    if not h or not t or h.group(1) != kernel_source_hash():
        return None
    return int(t.group(1))


class ClockSampler:
    """SM clock and throttle reasons sampled while the GPU works: through NVML (the
    driver's library, read-only queries) every 2 ms in a thread when it loads, else
    through `nvidia-smi -lms 50`.  A timed region of a few milliseconds then still holds
    samples of its own."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    # NVML clock-event reason bits, in the order of REASONS
    NVML_BITS = (0x8, 0x40, 0x20, 0x4)

    def __init__(self, gpu_index: int, period_s: float = 0.002):
        self.gpu_index = gpu_index
        self.period_s = period_s
        self.proc = None
        self.path = None
        self.thread = None
        self.rows = []
        self.source = "none"
        self._stop = False

    def _nvml(self):
        import ctypes

        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return None
        if lib.nvmlInit_v2() != 0:
            return None
        handle = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu_index), ctypes.byref(handle)) != 0:
            return None
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
        mx = ctypes.c_uint()
        if reasons is None or lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) != 0:
            return None
        return lib, handle, reasons, float(mx.value)

    def _loop(self, lib, handle, reasons, max_mhz):
        import ctypes

        clk, bits = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop:
            ok = lib.nvmlDeviceGetClockInfo(handle, 1, ctypes.byref(clk)) == 0 and \
                reasons(handle, ctypes.byref(bits)) == 0
            if ok:
                flags = ["Active" if bits.value & b else "Not Active" for b in self.NVML_BITS]
                self.rows.append((time.time(), float(clk.value), max_mhz, flags))
            time.sleep(self.period_s)

    def start(self):
        import threading

        nv = self._nvml()
        if nv is not None:
            self.source = "nvml every %.0f ms" % (self.period_s * 1e3)
            self.thread = threading.Thread(target=self._loop, args=nv, daemon=True)
            self.thread.start()
            time.sleep(0.05)
            return
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            self.source = "nvidia-smi every 50 ms"
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.thread is not None:
            self._stop = True
            self.thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def _smi_rows(self):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
                except ValueError:
                    continue
            os.unlink(self.path)
        return rows

    def summary(self, t0: float, t1: float):
        rows = list(self.rows) if self.thread is not None else self._smi_rows()
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "none",
                    "source": self.source}
        inside = [r for r in rows if t0 <= r[0] <= t1]
        window = "timed"
        if len(inside) < 3:
            inside = [r for r in rows if r[0] <= t1 + 0.2]
            window = "warmup+timed"
        reasons = sorted({name for r in inside for name, v in zip(self.REASONS, r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window, "source": self.source}


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over all ranks (the slowest rank's time); x itself when alone."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(world: int, tokens_per_rank: int, ms_per_step: float) -> float:
    """Weak scaling: every rank processes its own pack of tokens_per_rank tokens."""
    return world * tokens_per_rank / (ms_per_step / 1e3)


def cp_tokens_per_s(world: int, pack_tokens: int, rank_tokens: int, ms_per_step: float) -> float:
    """Strong scaling of one pack over a context-parallel group: the pack's tokens over
    the slowest rank's step time; on one GPU (an emulated rank) that rank's own tokens."""
    return (pack_tokens if world > 1 else rank_tokens) / (ms_per_step / 1e3)


def physical_gpu_index(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [v for v in vis.split(",") if v.strip()]
    if ids and local_rank < len(ids) and ids[local_rank].strip().isdigit():
        return int(ids[local_rank])
    return local_rank


# ---------------------------------------------------------------- reference arm (CPU oracle)

def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import numpy as np

    import oracle
    from packed_varlen_rope_gb300 import shards as shp
    from packed_varlen_rope_gb300 import workloads as wl

    oracle.build()
    w = wl.WORKLOADS[args.workload]
    if args.layout != "packed" and w.padded_samples is None:
        print("--layout %s needs a workload with padded samples (3)" % args.layout, file=sys.stderr)
        return 2
    # the pack, layout and context-parallel shard our arm times, so that both lines carry
    # the same config; the oracle is timed on consecutive rows of it
    pack = wl.make_pack(w, "packed" if args.layout == "packed" else "padded", rank=0)
    cp, shards, segs, rank_tokens = args.cp_size, None, None, None
    if cp > 1:
        if args.layout != "packed" or not 0 <= args.cp_rank < cp:
            print("--cp-size needs the packed layout and 0 <= --cp-rank < --cp-size", file=sys.stderr)
            return 2
        shards = shp.cp_shards(pack.total_tokens, cp, args.cp_rank, load_balanced=True)
        segs = shp.shard_segments(shards)
        rank_tokens = sum(1 for r in shp.shard_rows(shards) if r < pack.total_tokens)
    pos = oracle.positions(pack.cu_seqlens, pack.total_tokens)
    if cp > 1:                                            # the rank's own rows, padding left out
        pos = pos[np.array([r for r in shp.shard_rows(shards) if r < pack.total_tokens], dtype=np.int64)]
    import torch

    def bits(shape, kind):
        t = wl.normal_bf16(shape, wl.seed(args.workload, kind), device="cpu")
        return t.view(torch.int16).numpy().view(np.uint16)

    def step(a, n):
        idx = np.arange(a, a + n) % len(pos)
        p = pos[idx]
        oracle.rope_rows(qs[:n], p, w.theta)
        oracle.rope_rows(ks[:n], p, w.theta)
        oracle.rope_rows(qs[:n], p, w.theta, bwd=True)
        oracle.rope_rows(ks[:n], p, w.theta, bwd=True)

    cal = 64
    qs = bits((4096, w.n_q_heads, w.head_dim), "q")
    ks = bits((4096, w.n_kv_heads, w.head_dim), "k")
    t = time.perf_counter()
    step(0, cal)
    per_token = (time.perf_counter() - t) / cal
    n = int(max(1, min(4096, args.reference_seconds / max(1, args.steps + args.warmup) / per_token)))
    a = 0
    for _ in range(args.warmup):
        step(a, n)
        a += n
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(a, n)
        a += n
    el = time.perf_counter() - t0
    value = args.steps * n / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16",
        "data": "synthetic",
        "config": rope_config(args, w, pack, world, args.cp_rank if cp > 1 else 0, shards, segs, rank_tokens),
        "reference_tokens_per_step": n,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "%d consecutive tokens of the %s pack%s per step (fwd+bwd of Q and K)"
                                   % (n, w.name, " (this rank's rows)" if cp > 1 else "")},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
        # the same oracle calls split over every host core, beside the single-core figure
        "cpu_baseline_all_cores": cpu_all_cores(w, pos[np.arange(qs.shape[0]) % len(pos)], qs, ks, qs,
                                                ks),
    }
    print(json.dumps(line), flush=True)
    return 0


def rope_config(args, w, pack, world, cp_rank=0, shards=None, segs=None, rank_tokens=None):
    """The workload description both arms print as ``config`` (the same keys and values
    for the same arguments): shape, pack, layout, parallelism, L2 note and cos/sin
    source."""
    import numpy as np

    cp = args.cp_size
    rank_tokens = pack.valid_tokens if rank_tokens is None else rank_tokens
    rows_moved = pack.total_tokens if args.layout == "padded" else rank_tokens
    bytes_per_pass = 4 * (w.n_q_heads + w.n_kv_heads) * w.head_dim * rows_moved
    span = int(np.max(np.diff(pack.cu_seqlens)))
    return {
        "workload": w.name, "total_tokens": pack.total_tokens, "valid_tokens": pack.valid_tokens,
        "n_seqs": pack.n_seqs, "max_seq_len": max(pack.lengths), "n_q_heads": w.n_q_heads,
        "n_kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "theta": w.theta,
        "layout": {"packed": "packed [T, H, d] bf16, in place",
                   "padded": "padded batch [B*pad_to, H, d] bf16, every row rotated, in place",
                   "padded-seq-used": "padded batch [B*pad_to, H, d] bf16, pad rows skipped (seq_used)"
                   }[args.layout],
        "valid_fraction": valid_fraction(pack),
        "parallelism": ("cp%d (rank %d of a load-balanced context-parallel group%s)"
                        % (cp, cp_rank, "" if world > 1 else ", emulated on one GPU")
                        if cp > 1 else "dp%d (independent packs)" % world),
        "l2": l2_note(bytes_per_pass, buffer_sets(bytes_per_pass)),
        "cp_shards": None if cp <= 1 else {"token_start_rows": shards, "segments": segs,
                                           "rank_tokens": rank_tokens},
        "cos_sin": ("evaluated per tile, no cache (binary32 double-float; binary64 where the rounding "
                    "is undecided)" if args.no_cache else
                    "fp32 cache of %d positions built once before timing" % span),
    }


def valid_fraction(pack) -> float:
    """Share of the rows that hold tokens: 1 for a pack, sum(L_b) / (B * pad_to) for a
    padded batch (the padding waste of the unsloth.ai page, section "Pourquoi le
    remplissage est-il nécessaire")."""
    return pack.valid_tokens / pack.total_tokens


def cpu_baseline(args, w, pack, q_sample, k_sample, dq_sample, dk_sample, skip_pad=False, pos=None):
    """The oracle as it stands, single-threaded, on a contiguous token sample (rows of a
    padded batch left out when ``skip_pad``, as the seq_used form leaves them).  ``pos``:
    the rows' positions when they are not the pack's tokens in order (a context-parallel
    rank's rows)."""
    import numpy as np

    import oracle

    oracle.build()
    if pos is None:
        pos = oracle.positions(pack.cu_seqlens, pack.total_tokens)
    if skip_pad and pack.valid_mask is not None:
        pos = np.where(pack.valid_mask, pos, -1).astype(np.int32)
    n_all = q_sample.shape[0]

    def run(n):
        p = pos[:n]
        return (oracle.rope_rows(q_sample[:n], p, w.theta), oracle.rope_rows(k_sample[:n], p, w.theta),
                oracle.rope_rows(dq_sample[:n], p, w.theta, bwd=True),
                oracle.rope_rows(dk_sample[:n], p, w.theta, bwd=True))

    cal = min(256, n_all)
    t = time.perf_counter()
    run(cal)
    per_token = (time.perf_counter() - t) / cal
    n = int(max(cal, min(n_all, args.cpu_seconds / per_token)))
    t = time.perf_counter()
    outputs = run(n)
    passes = 1
    while time.perf_counter() - t < 0.9 * args.cpu_seconds:   # the whole sample is quick: repeat it
        run(n)
        passes += 1
    el = time.perf_counter() - t
    valid = int(np.count_nonzero(pos[:n] >= 0)) if pack.valid_mask is None or skip_pad else \
        int(np.count_nonzero(pack.valid_mask[:n]))
    return {"value": passes * valid / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "first %d rows (%d tokens) of the %s batch, fwd+bwd of Q and K, %d pass(es) in %.1f s on "
                      "one host core" % (n, valid, w.name, passes, el)}, outputs, \
        cpu_all_cores(w, pos[:n], q_sample[:n], k_sample[:n], dq_sample[:n], dk_sample[:n], valid=valid)


def cpu_all_cores(w, pos, q, k, dq, dk, seconds=2.0, valid=None):
    """The same oracle calls split into equal token ranges, one per host core the
    process may run on (the C calls release the GIL), repeated for about `seconds`."""
    import concurrent.futures as cf

    import numpy as np

    import oracle

    cores = len(os.sched_getaffinity(0))
    n = q.shape[0]
    bounds = np.linspace(0, n, cores + 1).astype(np.int64)

    def part(i):
        lo, hi = bounds[i], bounds[i + 1]
        p = pos[lo:hi]
        oracle.rope_rows(q[lo:hi], p, w.theta)
        oracle.rope_rows(k[lo:hi], p, w.theta)
        oracle.rope_rows(dq[lo:hi], p, w.theta, bwd=True)
        oracle.rope_rows(dk[lo:hi], p, w.theta, bwd=True)

    reps = 0
    with cf.ThreadPoolExecutor(cores) as ex:
        t = time.perf_counter()
        while True:
            list(ex.map(part, range(cores)))
            reps += 1
            el = time.perf_counter() - t
            if el >= seconds:
                break
    return {"value": reps * (n if valid is None else valid) / el, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "first %d tokens of the %s pack in %d token ranges on %d threads, %d passes in %.1f s"
                      % (n, w.name, cores, cores, reps, el)}


def parity_block(gpu_outputs, oracle_outputs, inputs):
    """Element-by-element comparison of the timed launch configuration's results with
    the oracle on the CPU-baseline sample: counts of differing bf16 elements and the
    largest difference in bf16 units in the last place."""
    import numpy as np

    n_el = mism = 0
    max_ulp = 0
    for got, ref, _x in zip(gpu_outputs, oracle_outputs, inputs):
        g = got[: ref.shape[0]]
        n_el += g.size
        diff = g != ref
        mism += int(np.count_nonzero(diff))
        if diff.any():
            gi = g[diff].astype(np.int32)
            ri = ref[diff].astype(np.int32)
            to_ordered = lambda b: np.where(b & 0x8000, 0x8000 - (b & 0x7FFF), 0x8000 + b)  # noqa: E731
            max_ulp = max(max_ulp, int(np.abs(to_ordered(gi) - to_ordered(ri)).max()))
    return {"elements": n_el, "bit_mismatch": mism, "max_bf16_ulp": max_ulp,
            "bar": "<= 2 bf16 ULP and <= 1e-2 (tests/parity_util.py); expected bit-identical"}


# ---------------------------------------------------------------- our arm

def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    from packed_varlen_rope_gb300 import build as _build

    _build.build()
    import packed_varlen_rope_gb300 as pr
    from packed_varlen_rope_gb300 import workloads as wl

    # the rank's GPU is made current before the process group exists, so that NCCL's
    # communicator and every barrier use it
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    w = wl.WORKLOADS[args.workload]
    if args.layout != "packed" and w.padded_samples is None:
        print("--layout %s needs a workload with padded samples (3)" % args.layout, file=sys.stderr)
        return 2
    cp = args.cp_size
    if cp > 1 and (args.layout != "packed" or (world > 1 and world != cp) or not 0 <= args.cp_rank < cp):
        print("--cp-size needs the packed layout, as many ranks as the group size under torchrun, and "
              "0 <= --cp-rank < --cp-size", file=sys.stderr)
        return 2
    cp_rank = (rank if world > 1 else args.cp_rank) if cp > 1 else 0
    seed_rank = 0 if cp > 1 else rank                    # context parallelism: one pack for all ranks
    pack = wl.make_pack(w, "packed" if args.layout == "packed" else "padded", rank=seed_rank)
    T = pack.total_tokens
    if args.layout != "packed":
        n_b, _, _, pad_to = w.padded_samples
        assert abs(valid_fraction(pack) - sum(pack.lengths) / (n_b * pad_to)) < 1e-12
    span = int(np.max(np.diff(pack.cu_seqlens)))          # longest sample, pad rows included
    shape_q, shape_k = (T, w.n_q_heads, w.head_dim), (T, w.n_kv_heads, w.head_dim)
    q = wl.normal_bf16(shape_q, wl.seed(args.workload, "q", seed_rank), device=dev)
    k = wl.normal_bf16(shape_k, wl.seed(args.workload, "k", seed_rank), device=dev)
    dq = wl.normal_bf16(shape_q, wl.seed(args.workload, "dq", seed_rank), device=dev)
    dk = wl.normal_bf16(shape_k, wl.seed(args.workload, "dk", seed_rank), device=dev)
    segs = shards = None
    rank_tokens = pack.valid_tokens                       # tokens this rank rotates per pass
    if cp > 1:
        # this rank's chunks, one after the other in its own buffers (padding rows past the
        # pack's end stay zero and lie outside every sample)
        shards = pr.cp_shards(T, cp, cp_rank, load_balanced=True)
        segs = pr.shard_segments(shards)
        rows = torch.tensor(pr.shard_rows(shards), device=dev)
        inside = rows < T
        rank_tokens = int(inside.sum())

        def rank_rows(t):
            out = torch.zeros((rows.numel(),) + tuple(t.shape[1:]), dtype=t.dtype, device=dev)
            out[inside] = t[rows[inside]]
            return out

        q, k, dq, dk = (rank_rows(t) for t in (q, k, dq, dk))
        T = rows.numel()
        shape_q, shape_k = (T, w.n_q_heads, w.head_dim), (T, w.n_kv_heads, w.head_dim)
        local_rows = rows.cpu().numpy()
    cu = torch.from_numpy(pack.cu_seqlens).to(dev)
    cache = None if args.no_cache else pr.new_cos_sin_cache(span, w.head_dim, w.theta, device=dev)
    stream = torch.cuda.current_stream(dev)
    used = torch.tensor(pack.lengths, dtype=torch.int32, device=dev) if args.layout == "padded-seq-used" else None

    def fwd(a, b):
        if used is None and segs is None:
            pr.rope_qk_fwd(a, b, cu, w.theta, cos_sin_cache=cache)
        else:
            pr.rope_qk_apply(a, b, w.theta, cu_seqlens=cu, seq_used=used, segments=segs, cos_sin_cache=cache)

    def bwd(a, b):
        if used is None and segs is None:
            pr.rope_qk_bwd(a, b, cu, w.theta, cos_sin_cache=cache)
        else:
            pr.rope_qk_apply(a, b, w.theta, cu_seqlens=cu, seq_used=used, segments=segs, cos_sin_cache=cache,
                             backward=True)

    do_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    samples = None
    to_np = lambda t, n: t[:n].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)  # noqa: E731
    if do_cpu:
        # untouched device copies of the inputs, for the oracle samples and the parity
        # check after the timed regions (the host copies are taken only then: freshly
        # written pageable host memory next to the e2e leg stalled its enqueueing thread)
        pristine = [t.clone() for t in (q, k, dq, dk)]
    # the e2e leg's pinned host inputs and outputs, allocated and filled here, well before
    # that leg runs, and with no pageable staging copy
    e2e_bufs = None if args.no_e2e else pinned_buffers(q, k, dq, dk)

    rows_moved = T if args.layout == "padded" else rank_tokens     # rows one launch reads and writes
    bytes_per_pass = 4 * (w.n_q_heads + w.n_kv_heads) * w.head_dim * rows_moved
    # the kernel instance the library dispatches for this call (head_dim template, 64-bit offsets)
    launch = pr.rope_qk_launch_info(q, k, w.theta, cu_seqlens=cu, cos_sin_cache=cache, seq_used=used,
                                    segments=segs)

    # a small pack's tensors could stay in L2 from one step to the next: the steps cycle
    # through enough copies that a launch's inputs were last touched 4 x L2 bytes ago
    n_sets = buffer_sets(bytes_per_pass)
    sets = [(q, k, dq, dk)] + [tuple(t.clone() for t in (q, k, dq, dk)) for _ in range(n_sets - 1)]

    sampler = ClockSampler(physical_gpu_index(local))
    sampler.start()
    for i in range(max(3, args.warmup)):
        sq, sk, sdq, sdk = sets[i % n_sets]
        fwd(sq, sk)
        bwd(sdq, sdk)
    torch.cuda.synchronize()

    # Only the two events around the region: an event recorded between two launches
    # would order the second after the first's completion and take away the overlap of
    # back-to-back launches (programmatic dependent launch); the mean launch time is the
    # region's duration over its launches, gaps included.
    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start.record(stream)
    for i in range(K):
        sq, sk, sdq, sdk = sets[i % n_sets]
        fwd(sq, sk)
        bwd(sdq, sdk)
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t_wall1 = time.time()
    sampler.stop()
    total_ms = start.elapsed_time(end)
    del sets
    avg_launch_s = total_ms / (2 * K) / 1e3          # this rank's mean time per launch
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / K
    if cp > 1:
        # one pack split over the group: the pack's tokens over the slowest rank's time
        # (one GPU: the emulated rank's own tokens)
        value = cp_tokens_per_s(world, pack.valid_tokens, rank_tokens, ms_per_step)
    else:
        value = whole_job_tokens_per_s(world, pack.valid_tokens, ms_per_step)
    achieved = bytes_per_pass / avg_launch_s / 1e9
    peak, peak_kind = measured_peak()
    clocks = sampler.summary(t_wall0, t_wall1)

    copy_ref = size_matched_copy(torch, dev, bytes_per_pass, n_sets, 2 * K)
    copy_ref["frac_of_measured"] = copy_ref["gbs"] / peak
    copy_ref["launch_time_over_copy_time"] = avg_launch_s * 1e6 / copy_ref["us_per_copy"]

    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(args, pr, w, pack, e2e_bufs, cu, cache, stream, world, dev, used, segs,
                         pack.valid_tokens if cp > 1 and world > 1 else rank_tokens, scale_world=cp == 1)
        del e2e_bufs

    cpu = parity = None
    if do_cpu:
        samples = tuple(to_np(t, min(T, 65536)) for t in pristine)
        pos_override = None
        if cp > 1:
            import oracle

            oracle.build()
            pos_override = oracle.positions(pack.cu_seqlens, max(pack.total_tokens, int(local_rows.max()) + 1))
            pos_override = pos_override[local_rows].astype(np.int32)
        cpu, ref_outputs, cpu_all = cpu_baseline(args, w, pack, *samples, skip_pad=used is not None,
                                                 pos=pos_override)
        pq, pk, pdq, pdk = pristine
        fwd(pq, pk)
        bwd(pdq, pdk)
        torch.cuda.synchronize()
        n = ref_outputs[0].shape[0]
        parity = parity_block([to_np(t, n) for t in (pq, pk, pdq, pdk)], ref_outputs, samples)
        del pristine, pq, pk, pdq, pdk

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "strong" if cp > 1 else "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16",
        "data": "synthetic",
        "config": rope_config(args, w, pack, world, cp_rank, shards, segs, rank_tokens),
        "hbm_gbs": 2 * bytes_per_pass / (ms_per_step / 1e3) / 1e9,
        "hbm_frac_of_measured": 2 * bytes_per_pass / (ms_per_step / 1e3) / 1e9 / peak,
        "hbm_frac_of_nominal_8tbs": 2 * bytes_per_pass / (ms_per_step / 1e3) / 1e9 / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     # the profiled launch is the whole packed pack with a cache: a CP
                     # rank's launch (half the rows) or another layout has no capture
                     "traffic": (profiled_traffic(w.name) if cache is not None and args.layout == "packed"
                                 and cp == 1 else None),
                     "kernel": launch.kernel_name(),
                     "grid": {"ctas": launch.grid, "threads": launch.threads, "tile_tokens": launch.tile_tokens},
                     "algorithmic_bytes_per_launch": bytes_per_pass,
                     "avg_launch_us": avg_launch_s * 1e6, "peak_kind": peak_kind + " (hbm_gbs)"},
        "size_matched_copy": copy_ref,
        "clocks": clocks,
        "gpu_launches": 2 * K,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if cpu is not None:
        line["cpu_baseline"] = cpu
        line["cpu_baseline_all_cores"] = cpu_all
        line["parity"] = parity
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def pinned_buffers(*tensors):
    """(inputs, outputs): pinned host copies of device tensors and pinned host tensors of
    the same shapes, each allocated pinned directly (no pageable staging copy)."""
    import torch

    host = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in tensors]
    for h, t in zip(host, tensors):
        h.copy_(t)
    work = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in tensors]
    return host, work


def end_to_end(args, pr, w, pack, bufs, cu, cache, stream, world, dev, used=None, segs=None,
               tokens=None, scale_world=True):
    """Same metric through the public host-buffer call (rope_qk_host) with the inputs in
    pinned host memory (``bufs`` from ``pinned_buffers(q, k, dq, dk)``): every step
    streams Q, K (forward) and dQ, dK (backward) from the host through a device
    workspace in chunks and back, copies overlapped with the rotation; the results are
    complete in host memory when the step's stream ends."""
    import torch

    host, work = bufs
    per_token = (w.n_q_heads + w.n_kv_heads) * w.head_dim * 2
    rows = host[0].shape[0]
    tokens = pack.valid_tokens if tokens is None else tokens
    per_s = (lambda ms: whole_job_tokens_per_s(world, tokens, ms)) if scale_world else \
        (lambda ms: tokens / (ms / 1e3))  # noqa: E731
    chunk = max(8, (rows // 16) // 8 * 8)
    ws = torch.empty(2 * chunk * per_token + 4096, dtype=torch.uint8, device=dev)
    h2d = sum(t.numel() * t.element_size() for t in host)

    def step():
        pr.rope_qk_host(host[0], host[1], w.theta, ws, cu_seqlens=cu, cos_sin_cache=cache,
                        q_out=work[0], k_out=work[1], seq_used=used, segments=segs)
        pr.rope_qk_host(host[2], host[3], w.theta, ws, cu_seqlens=cu, cos_sin_cache=cache, backward=True,
                        q_out=work[2], k_out=work[3], seq_used=used, segments=segs)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    E = max(1, args.e2e_steps)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(E + 1)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    marks[0].record(stream)
    for i in range(E):
        step()
        marks[i + 1].record(stream)
    torch.cuda.synchronize()
    steps_ms = [marks[i].elapsed_time(marks[i + 1]) for i in range(E)]
    ms = max_over_ranks(marks[0].elapsed_time(marks[E]) / E, world, dev)

    # The same step captured once in a CUDA graph and replayed: whole steps are queued
    # ahead, so a pause of the host thread (the host is shared) does not leave the GPU
    # idle; every replay still copies the inputs in from and the results out to pinned
    # host memory.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    g0.record(stream)
    for _ in range(E):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    gms = max_over_ranks(g0.elapsed_time(g1) / E, world, dev)
    return {"value": per_s(ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": h2d, "ms_per_step": ms, "steps": E,
            "step_ms_min": min(steps_ms), "step_ms_median": statistics.median(steps_ms),
            "step_ms_p90": sorted(steps_ms)[int(0.9 * (len(steps_ms) - 1))],
            "step_ms_max": max(steps_ms), "step_ms_max_index": steps_ms.index(max(steps_ms)),
            "steps_over_twice_median": sum(1 for t in steps_ms if t > 2 * statistics.median(steps_ms)),
            "path": "rope_qk_host: pinned host buffers streamed in %d-token chunks" % chunk,
            "graph_replay": {"value": per_s(gms), "ms_per_step": gms,
                             "steps": E, "path": "the same rope_qk_host calls captured in one CUDA graph"}}


def run_glu(args, rank, world, local):
    """SwiGLU / GeGLU forward + backward on one matrix shape (second workload of the
    source page: the MLP activation kernels with int64 indexing).  One step = glu_fwd
    (h = act(e) * g) then glu_bwd (de, dg into their own buffers)."""
    import torch

    from packed_varlen_rope_gb300 import build as _build

    _build.build()
    import packed_varlen_rope_gb300 as pr
    from packed_varlen_rope_gb300 import workloads as wl

    # the rank's GPU is made current before the process group exists, so that NCCL's
    # communicator and every barrier use it
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    w = wl.GLU_WORKLOADS[args.glu_workload]
    if args.glu_kind is not None:
        w = wl.GluWorkload(w.name, w.rows, w.cols, args.glu_kind, w.description)
    shape = (w.rows, w.cols)
    e = wl.normal_bf16(shape, 7001 + rank * wl.RANK_SEED_STRIDE, device=dev)
    g = wl.normal_bf16(shape, 7002 + rank * wl.RANK_SEED_STRIDE, device=dev)
    dh = wl.normal_bf16(shape, 7003 + rank * wl.RANK_SEED_STRIDE, device=dev)
    h, de, dg = (torch.empty(shape, dtype=torch.bfloat16, device=dev) for _ in range(3))
    stream = torch.cuda.current_stream(dev)
    n = w.rows * w.cols
    fwd_bytes, bwd_bytes = 6 * n, 10 * n
    for _ in range(max(3, args.warmup)):
        pr.glu_fwd(w.kind, e, g, h)
        pr.glu_bwd(w.kind, dh, e, g, de, dg)
    sampler = ClockSampler(physical_gpu_index(local))
    sampler.start()
    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    start.record(stream)
    for _ in range(K):                       # no events between launches (they would serialise them)
        pr.glu_fwd(w.kind, e, g, h)
        pr.glu_bwd(w.kind, dh, e, g, de, dg)
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t1 = time.time()
    sampler.stop()
    ms = max_over_ranks(start.elapsed_time(end), world, dev) / K

    def per_launch(fn, n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n / 1e3

    # each kernel on its own, back to back, for the per-kernel rooflines
    n_each = max(3, K // 2)
    fwd_s = per_launch(lambda: pr.glu_fwd(w.kind, e, g, h), n_each)
    bwd_s = per_launch(lambda: pr.glu_bwd(w.kind, dh, e, g, de, dg), n_each)
    peak, peak_kind = measured_peak()
    if rank == 0:
        line = {
            "metric": "SwiGLU/GeGLU fwd+bwd tokens/s and HBM GB/s", "value": whole_job_tokens_per_s(world, w.rows, ms),
            "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.name, "rows": w.rows, "cols": w.cols, "kind": w.kind,
                       "l2": "no flush: %.1f GB per step > 129 MB L2" % ((fwd_bytes + bwd_bytes) / 1e9)},
            "hbm_gbs": (fwd_bytes + bwd_bytes) / (ms / 1e3) / 1e9,
            "roofline": {"bound": "hbm", "unit": "GB/s", "peak": peak, "peak_kind": peak_kind + " (hbm_gbs)",
                         "timing": "each kernel launched %d times back to back after the step region, "
                                   "CUDA events around the run" % n_each,
                         "kernels": {
                             "glu_fwd": {"achieved": fwd_bytes / fwd_s / 1e9, "frac": fwd_bytes / fwd_s / 1e9 / peak,
                                         "algorithmic_bytes_per_launch": fwd_bytes, "avg_launch_us": fwd_s * 1e6},
                             "glu_bwd": {"achieved": bwd_bytes / bwd_s / 1e9, "frac": bwd_bytes / bwd_s / 1e9 / peak,
                                         "algorithmic_bytes_per_launch": bwd_bytes, "avg_launch_us": bwd_s * 1e6}}},
            "clocks": sampler.summary(t0, t1),
            "gpu_launches": 2 * K,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_rope_forms(args, rank, world, local):
    """The forward rotation of one workload through each input form of the C ABI: the
    median time per launch (or per group of launches, for shards), algorithmic GB/s and
    its fraction of the measured copy rate, and a check of the result -- bit-identical
    to the contiguous path where the form computes the same thing, and against the
    oracle on seeded sample tokens for the rescaled rotation."""
    import numpy as np
    import torch

    from packed_varlen_rope_gb300 import build as _build

    _build.build()
    import packed_varlen_rope_gb300 as pr
    from packed_varlen_rope_gb300 import workloads as wl

    if rank != 0:
        return 0
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = wl.WORKLOADS[args.workload]
    pack = wl.make_pack(w)
    T, Hq, Hkv, d = pack.total_tokens, w.n_q_heads, w.n_kv_heads, w.head_dim
    q0 = wl.normal_bf16((T, Hq, d), wl.seed(w.index, "q"), device=dev)
    k0 = wl.normal_bf16((T, Hkv, d), wl.seed(w.index, "k"), device=dev)
    cu = torch.from_numpy(pack.cu_seqlens).to(dev)
    rows = max(pack.lengths)
    cache = pr.new_cos_sin_cache(rows, d, w.theta, device=dev)
    q_ref, k_ref = q0.clone(), k0.clone()
    pr.rope_qk_fwd(q_ref, k_ref, cu, w.theta, cos_sin_cache=cache)
    nbytes = 4 * (Hq + Hkv) * d * pack.valid_tokens
    peak, peak_kind = measured_peak()
    bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)  # noqa: E731

    # read before every timed replay, so that no form finds its tensors in L2 (a read
    # leaves clean lines: no write-back lands in the timed replay)
    flush = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def timed(fn, reps=50):
        # each form captured once in a CUDA graph and replayed, so that groups of short
        # launches (the shard forms) are timed without the host's launch gaps
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(3):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        for _ in range(3):
            graph.replay()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda.synchronize()
        for a, b in ev:
            flush.sum()
            a.record()
            graph.replay()
            b.record()
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ev) / 1e3

    def same(q, k):
        return "bit-identical to contiguous" if torch.equal(q, q_ref) and torch.equal(k, k_ref) else "MISMATCH"

    forms = {}

    def record(name, fn, check, launches=1, nbytes_form=None):
        sec = timed(fn)
        nb = nbytes if nbytes_form is None else nbytes_form
        forms[name] = {"us": sec * 1e6, "gbs": nb / sec / 1e9, "frac": nb / sec / 1e9 / peak,
                       "launches": launches, "bytes": nb, "check": check}

    # contiguous [T, H, d]
    q, k = q0.clone(), k0.clone()
    pr.rope_qk_fwd(q, k, cu, w.theta, cos_sin_cache=cache)
    record("contiguous [T,H,d], rope_qk_fwd", lambda: pr.rope_qk_fwd(q, k, cu, w.theta, cos_sin_cache=cache),
           same(q, k))
    # Q and K slices of one fused [T, Hq + 2 Hkv, d] QKV output
    qkv = torch.empty((T, Hq + 2 * Hkv, d), dtype=torch.bfloat16, device=dev)
    qkv[:, :Hq].copy_(q0)
    qkv[:, Hq:Hq + Hkv].copy_(k0)
    qkv[:, Hq + Hkv:].fill_(1.5)
    qs, ks = qkv[:, :Hq], qkv[:, Hq:Hq + Hkv]
    pr.rope_qk_apply(qs, ks, w.theta, cu_seqlens=cu, cos_sin_cache=cache)
    check = same(qs, ks) + ("" if torch.all(qkv[:, Hq + Hkv:] == 1.5) else ", V CHANGED")
    record("fused QKV slices in place, rope_qk_apply",
           lambda: pr.rope_qk_apply(qs, ks, w.theta, cu_seqlens=cu, cos_sin_cache=cache), check)
    del qkv, qs, ks
    # head-major [H, T, d] storage, passed as [T, H, d] views
    qh = q0.transpose(0, 1).contiguous().transpose(0, 1)
    kh = k0.transpose(0, 1).contiguous().transpose(0, 1)
    pr.rope_qk_apply(qh, kh, w.theta, cu_seqlens=cu, cos_sin_cache=cache)
    record("head-major [H,T,d] views, rope_qk_apply",
           lambda: pr.rope_qk_apply(qh, kh, w.theta, cu_seqlens=cu, cos_sin_cache=cache), same(qh, kh))
    del qh, kh
    # out of place
    q, k = q0.clone(), k0.clone()
    qo, ko = torch.empty_like(q0), torch.empty_like(k0)
    pr.rope_qk_apply(q, k, w.theta, cu_seqlens=cu, cos_sin_cache=cache, q_out=qo, k_out=ko)
    check = same(qo, ko) + ("" if torch.equal(q, q0) and torch.equal(k, k0) else ", INPUT CHANGED")
    record("out of place, rope_qk_apply",
           lambda: pr.rope_qk_apply(q, k, w.theta, cu_seqlens=cu, cos_sin_cache=cache, q_out=qo, k_out=ko), check)
    del qo, ko
    # explicit position ids
    pos = pr.rope_qk_positions(cu, T)
    q, k = q0.clone(), k0.clone()
    pr.rope_qk_apply(q, k, w.theta, position_ids=pos, cos_sin_cache=cache)
    record("position_ids int32 [T], rope_qk_apply",
           lambda: pr.rope_qk_apply(q, k, w.theta, position_ids=pos, cos_sin_cache=cache), same(q, k))
    # context-parallel shards, cp = 2.  Contiguous: rank r holds tokens [r T/2, (r+1) T/2)
    # of the one pack buffer (a token offset per launch).  Load-balanced: rank r holds
    # chunks r and 3 - r of 4, one after the other in its own buffer, rotated in one
    # launch through the segment list; each rank's launch is timed alone (what a rank of
    # a real context-parallel group runs) and the two ranks back to back.
    q, k = q0.clone(), k0.clone()
    halves = [(0, T // 2), (T // 2, T)]

    def contiguous_shards():
        for a, b in halves:
            pr.rope_qk_apply(q[a:b], k[a:b], w.theta, cu_seqlens=cu, token_offset=a, cos_sin_cache=cache)

    contiguous_shards()
    record("cp=2 contiguous shards, both ranks (token_offset, 2 launches)", contiguous_shards, same(q, k),
           launches=2)
    cp = 2
    ranks = []
    for r in range(cp):
        shards = pr.cp_shards(T, cp, r, load_balanced=True)
        rows_r = torch.tensor(pr.shard_rows(shards), device=dev)
        inside = rows_r < T                                   # rows past the pack's end are padding
        ql = torch.zeros((rows_r.numel(), Hq, d), dtype=torch.bfloat16, device=dev)
        kl = torch.zeros((rows_r.numel(), Hkv, d), dtype=torch.bfloat16, device=dev)
        ql[inside], kl[inside] = q0[rows_r[inside]], k0[rows_r[inside]]
        ranks.append((ql, kl, pr.shard_segments(shards), rows_r, inside))

    def rank_launch(r):
        ql, kl, segs, _, _ = ranks[r]
        pr.rope_qk_apply(ql, kl, w.theta, cu_seqlens=cu, segments=segs, cos_sin_cache=cache)

    def lb_check():
        ok = True
        for ql, kl, _, rows_r, inside in ranks:
            ok = ok and torch.equal(ql[inside], q_ref[rows_r[inside]]) and torch.equal(kl[inside], k_ref[rows_r[inside]])
        return "bit-identical to contiguous" if ok else "MISMATCH"

    for r in range(cp):
        rank_launch(r)
    check = lb_check()
    rank_bytes = [4 * (Hq + Hkv) * d * int(x[4].sum()) for x in ranks]
    record("cp=2 load-balanced, rank 0 alone: chunks 0,3 (segments, 1 launch)", lambda: rank_launch(0), check,
           nbytes_form=rank_bytes[0])
    record("cp=2 load-balanced, rank 1 alone: chunks 1,2 (segments, 1 launch)", lambda: rank_launch(1), check,
           nbytes_form=rank_bytes[1])
    record("cp=2 load-balanced, both ranks (segments, 2 launches)", lambda: [rank_launch(r) for r in range(cp)],
           check, launches=2)
    del ranks
    # cos/sin evaluated in the kernel (no cache)
    q, k = q0.clone(), k0.clone()
    pr.rope_qk_fwd(q, k, cu, w.theta)
    record("no cos/sin cache (evaluated per tile), rope_qk_fwd",
           lambda: pr.rope_qk_fwd(q, k, cu, w.theta), same(q, k))
    # linear position rescale, factor 4, with its own cache; oracle on sampled tokens
    import oracle

    oracle.build()
    cache4 = pr.new_cos_sin_cache(rows, d, w.theta, device=dev, position_scale=4.0)
    q, k = q0.clone(), k0.clone()
    pr.rope_qk_apply(q, k, w.theta, cu_seqlens=cu, position_scale=4.0, cos_sin_cache=cache4)
    pick = np.unique(np.random.Generator(np.random.PCG64(wl.seed(w.index, "rows"))).integers(0, T, 2048))
    pick_dev = torch.from_numpy(pick).to(dev)
    opos = oracle.positions(pack.cu_seqlens, T)[pick]
    n_el = mism = 0
    for got, src in ((q, q0), (k, k0)):
        ref = oracle.rope_rows(bits(src[pick_dev]), opos, w.theta, scale=4.0)
        g = bits(got[pick_dev])
        n_el += g.size
        mism += int(np.count_nonzero(g != ref))
    record("position_scale 4 (scaled cache), rope_qk_apply",
           lambda: pr.rope_qk_apply(q, k, w.theta, cu_seqlens=cu, position_scale=4.0, cos_sin_cache=cache4),
           "oracle on %d sampled tokens: %d elements, %d differ" % (pick.size, n_el, mism))
    line = {"metric": "QK-RoPE forward per input form", "unit": "GB/s", "workload": w.name,
            "algorithmic_bytes_per_launch": nbytes, "peak": peak, "peak_kind": peak_kind + " (hbm_gbs)",
            "timing": "median of 50 CUDA-graph replays of each form (CUDA events), inputs %.2f GB > L2"
                      % (nbytes / 2e9),
            "forms": forms}
    print(json.dumps(line), flush=True)
    bad = [n for n, f in forms.items() if "MISMATCH" in f["check"] or "CHANGED" in f["check"] or
           not f["check"].endswith(" 0 differ") and f["check"].startswith("oracle")]
    return 1 if bad else 0


HEAD_SHAPES = ((64, 8, 64), (64, 8, 80), (64, 8, 96), (64, 8, 128), (64, 8, 256), (32, 8, 128), (32, 32, 64),
               (32, 32, 96))


def run_rope_shapes(args, rank, world, local):
    """Forward + backward back to back on head shapes beyond the workloads' (Hq, Hkv, d):
    each shape gets enough tokens for about 2.4 GB per launch, packed from samples of
    1,024 tokens, theta 1e6, a cos/sin cache; the mean time per launch over the timed
    launches (CUDA events around them only) and 512 seeded rows of the forward checked
    against the oracle bit for bit."""
    import numpy as np
    import torch

    from packed_varlen_rope_gb300 import build as _build

    _build.build()
    import oracle
    import packed_varlen_rope_gb300 as pr
    from packed_varlen_rope_gb300 import workloads as wl

    if rank != 0:
        return 0
    oracle.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peak, peak_kind = measured_peak()
    theta, sample = 1.0e6, 1024
    bits = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)  # noqa: E731
    shapes = {}
    for hq, hkv, d in HEAD_SHAPES:
        per_token = 4 * (hq + hkv) * d
        T = (2_415_919_104 // per_token) // sample * sample
        cu_np = np.arange(0, T + 1, sample, dtype=np.int32)
        cu = torch.from_numpy(cu_np).to(dev)
        q = wl.normal_bf16((T, hq, d), 8100 + d, device=dev)
        k = wl.normal_bf16((T, hkv, d), 8200 + d, device=dev)
        dq = wl.normal_bf16((T, hq, d), 8300 + d, device=dev)
        dk = wl.normal_bf16((T, hkv, d), 8400 + d, device=dev)
        cache = pr.new_cos_sin_cache(sample, d, theta, device=dev)
        pick = np.unique(np.random.Generator(np.random.PCG64(8500 + d)).integers(0, T, 512))
        pick_dev = torch.from_numpy(pick).to(dev)
        q0, k0 = bits(q[pick_dev]), bits(k[pick_dev])
        pr.rope_qk_fwd(q, k, cu, theta, cos_sin_cache=cache)
        torch.cuda.synchronize()
        pos = (pick % sample).astype(np.int32)
        mism = int(np.count_nonzero(bits(q[pick_dev]) != oracle.rope_rows(q0, pos, theta))) + \
            int(np.count_nonzero(bits(k[pick_dev]) != oracle.rope_rows(k0, pos, theta)))
        n_el = q0.size + k0.size
        for _ in range(max(3, args.warmup)):
            pr.rope_qk_fwd(q, k, cu, theta, cos_sin_cache=cache)
            pr.rope_qk_bwd(dq, dk, cu, theta, cos_sin_cache=cache)
        K = max(10, min(args.steps, 200))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(K):
            pr.rope_qk_fwd(q, k, cu, theta, cos_sin_cache=cache)
            pr.rope_qk_bwd(dq, dk, cu, theta, cos_sin_cache=cache)
        b.record()
        torch.cuda.synchronize()
        sec = a.elapsed_time(b) / 1e3 / (2 * K)
        nbytes = per_token * T
        info = pr.rope_qk_launch_info(q, k, theta, cu_seqlens=cu, cos_sin_cache=cache)
        shapes["%d/%d/%d" % (hq, hkv, d)] = {
            "tokens": T, "us": sec * 1e6, "gbs": nbytes / sec / 1e9, "frac": nbytes / sec / 1e9 / peak,
            "kernel": info.kernel_name(), "tile_tokens": info.tile_tokens,
            "check": "oracle on %d sampled tokens: %d elements, %d differ" % (pick.size, n_el, mism)}
        del q, k, dq, dk, cache
        torch.cuda.empty_cache()
    line = {"metric": "QK-RoPE fwd+bwd per head shape (Hq/Hkv/d)", "unit": "GB/s", "peak": peak,
            "peak_kind": peak_kind + " (hbm_gbs)", "theta": theta, "sample_tokens": sample,
            "timing": "mean per launch over back-to-back forward and backward launches (CUDA events around them)",
            "shapes": shapes}
    print(json.dumps(line), flush=True)
    return 1 if any(not v["check"].endswith(" 0 differ") for v in shapes.values()) else 0


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.gpus != world and world == 1 and args.gpus > 1:
        print("--gpus %d needs torchrun with %d processes" % (args.gpus, args.gpus), file=sys.stderr)
        return 2
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.path == "glu":
        return run_glu(args, rank, world, local)
    if args.path == "rope-forms":
        return run_rope_forms(args, rank, world, local)
    if args.path == "rope-shapes":
        return run_rope_shapes(args, rank, world, local)
    return run_ours(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
