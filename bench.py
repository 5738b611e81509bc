#!/usr/bin/env python
"""Benchmark of the fused DSA decode step on one or more GB300s.

One step = the whole hot path over one batch through dsa_fused_decode: the lightning indexer with
on-chip Top-K followed by sparse flash attention over the selected rows.  At the default workload that
is one kernel launch (each token's indexer, Top-K and attention run in one thread-block cluster); shapes
the single-launch kernel does not serve take two launches (the attention kernel as a programmatic
dependent of the indexer).  The roofline is taken on the dominant launch, timed with CUDA events around
each launch in a second pass; a third pass times the separate dsa_indexer_topk / dsa_sparse_attn calls
for the per-kernel breakdown.  Default workload: decode, 32 sequences x 32768 cached tokens,
one query token each, indexer 64 heads x 128-d bf16, K = 2048, SFA 128 heads x 576-d bf16 (synthetic,
seeded; inputs larger than L2 so no flush is needed between steps).

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5] [--impl ours|reference]
For N > 1 launch one process per GPU (torch.distributed.run); every rank runs its own batch (weak
scaling, no collective on the data path) and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused DSA decode tokens/s at 32K ctx; achieved HBM GB/s vs GB300 peak"
UNIT = "tokens/s"


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=2, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--soak-s", type=float, default=1.0, help="seconds of untimed steps under clock sampling")
    ap.add_argument("--idx-mx", action="store_true",
                    help="MXFP8 indexer inputs (E4M3 codes, one E8M0 scale per 32 elements)")
    ap.add_argument("--kv-fp8", action="store_true",
                    help="latent-KV cache in the FP8 row layout (one scale per 128 elements of each token)")
    ap.add_argument("--no-prefill-indexer", action="store_true",
                    help="skip the prefill-chunk indexer measurement (the tensor-bound half of the path)")
    ap.add_argument("--clock-window-s", type=float, default=1.0,
                    help="seconds of back-to-back repeats of the timed steps, sampled for clocks")
    return ap.parse_args(argv)


# ------------------------------------------------------------------------------------------------------
# distributed plumbing (one process per GPU; gloo works for CPU tests)
# ------------------------------------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(world, backend):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value: float) -> float:
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64)
    if dist.get_backend() == "nccl":
        t = t.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, value: float) -> float:
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64)
    if dist.get_backend() == "nccl":
        t = t.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.samples = []  # (host time, sm_mhz, max_mhz, reasons set)
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", f"-lms={self.period}",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            reasons = {n for n, v in zip(names, parts[5:9]) if v.lower().startswith("active")}
            self.samples.append((time.time(), sm, mx, reasons))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed region"
        if not inside and self.samples:  # timed region shorter than the sampling period: nearest samples
            inside = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            window = "nearest samples to the timed region (soak + timed steps)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "unavailable"}
        reasons = sorted(set().union(*[s[3] for s in inside]))
        return {"sm_mhz": float(np.median([s[1] for s in inside])), "sm_max_mhz": max(s[2] for s in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


# ------------------------------------------------------------------------------------------------------
# algorithmic traffic (bytes each launch must move at minimum)
# ------------------------------------------------------------------------------------------------------
def indexer_bytes(wl) -> int:
    elem = 1 if wl.idx_fp8 else 2
    pos = wl.query_positions()
    # every query block reads its sequence's keys up to its last query position
    ctx = int(sum(int(wl.seq_lens[b]) for b in range(wl.batch)))
    kbytes = ctx * wl.idx_dim * elem + (ctx * 4 if wl.idx_fp8 else 0)
    pages = int(sum(math.ceil(int(L) / 64) for L in wl.seq_lens)) * 4
    qbytes = wl.total_q * wl.idx_heads * (wl.idx_dim * elem + 4 + (4 if wl.idx_fp8 else 0))
    out = wl.total_q * wl.top_k * 4
    del pos
    return kbytes + pages + qbytes + out


def sfa_bytes(wl, topk) -> int:
    sel = int((topk >= 0).sum())
    gather = sel * (wl.kv_cache.shape[-1] if getattr(wl, "kv_fp8", False) else wl.kv_dim * 2)
    qs = wl.total_q * wl.attn_heads * wl.kv_dim * 2
    out = wl.total_q * wl.attn_heads * (wl.v_dim * 2 + 4)
    idx = wl.total_q * wl.top_k * 4
    pages = 0
    seq = wl.query_seq()
    for t in range(wl.total_q):
        s = topk[t][topk[t] >= 0]
        pages += np.unique(s // 64).shape[0] * 4
    del seq
    return gather + qs + out + idx + pages


def indexer_flops(wl) -> int:
    """Algorithmic score flops: 2 * Hi * Di per (query, visible position)."""
    pos = wl.query_positions()
    return int(2 * wl.idx_heads * wl.idx_dim * int(np.sum(pos.astype(np.int64) + 1)))


# workloads whose indexer is bound by the tensor pipe rather than HBM (the prefill chunk: 4096 queries
# over 64K positions, 4.26 TFLOP of scores against 16.8 MB of keys)
TENSOR_BOUND_CONFIGS = (4,)


def workload_name(args) -> str:
    from gen.workloads import CONFIG_NAMES

    return (CONFIG_NAMES[args.config] + ("_mxfp8" if getattr(args, "idx_mx", False) else "") +
            ("_kvfp8" if getattr(args, "kv_fp8", False) else ""))


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# the source files each kernel is built from (a profile is valid only for the sources it was taken on)
KERNEL_SOURCES = {
    "indexer": ["indexer.cu", "indexer_impl.cuh", "common.cuh", "internal.h"],
    "sfa": ["sfa.cu", "sfa_impl.cuh", "common.cuh", "internal.h"],
    "decode": ["decode.cu", "indexer_impl.cuh", "sfa_impl.cuh", "common.cuh", "internal.h"],
}


def _code_only(text: str) -> str:
    """The source without // comments, trailing blanks and empty lines (the kernel sources use no block
    comments and no // inside string literals), so that a comment edit does not mark a profile stale."""
    lines = []
    for line in text.splitlines():
        i = line.find("//")
        if i >= 0:
            line = line[:i]
        line = line.rstrip()
        if line:
            lines.append(line)
    return "\n".join(lines)


def source_sha(kernel: str) -> str:
    """Hash of the code (comments excluded) of the files a kernel is built from."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "sparse_attention_dsa_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def kernel_traffic(kernel: str, profile_md: str):
    """dram bytes per launch from a committed ncu summary, if it was taken on the current kernel sources."""
    try:
        sha = source_sha(kernel)
        txt = open(os.path.join(ROOT, "profiles", profile_md)).read()
    except OSError:
        return None
    m_sha = re.search(r"source_sha256_16:\s*([0-9a-f]+)", txt)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m_sha or not m_b or m_sha.group(1) != sha:
        return None
    return float(m_b.group(1))


# ------------------------------------------------------------------------------------------------------
# the oracle on host cores (cpu_baseline leg and the reference arm)
# ------------------------------------------------------------------------------------------------------
def oracle_step(wl, tlist):
    import oracle

    topk, _, _ = oracle.indexer_topk(wl, tlist)
    oracle.sparse_attn(wl, topk, tlist)


def oracle_cores():
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


def cpu_baseline(wl, budget_s=20.0):
    """Oracle throughput on a bounded sample of the workload's query tokens (one token per core per round)."""
    cores = oracle_cores()
    n = min(wl.total_q, cores)
    tl = list(range(n))
    t0 = time.perf_counter()
    oracle_step(wl, tl)
    dt = time.perf_counter() - t0
    rounds = 1
    while time.perf_counter() - t0 + dt < budget_s and rounds * n < wl.total_q:
        tl = [(rounds * n + i) % wl.total_q for i in range(n)]
        oracle_step(wl, tl)
        rounds += 1
    total = time.perf_counter() - t0
    return {"value": rounds * n / total, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{rounds * n} of {wl.total_q} query tokens of the same workload (indexer + Top-K + "
                      f"attention, float64 C oracle, OpenMP over tokens), {total:.1f} s"}


def cpu_single_thread():
    """The oracle on one core: the 4K-context decode token and one sequence of the 32K-context decode."""
    import oracle
    from gen.workloads import config

    old = oracle.set_threads(1)
    res = {}
    try:
        for name, wl in (("decode_b1_ctx4096", config(1)), ("decode_ctx32768_one_sequence", config(2, batch=1))):
            t0 = time.perf_counter()
            oracle_step(wl, list(range(wl.total_q)))
            dt = time.perf_counter() - t0
            res[name] = {"value": wl.total_q / dt, "unit": UNIT, "seconds": dt}
    finally:
        oracle.set_threads(old)
    return {"cores": 1, "kind": "oracle", **res}


def run_reference(args, wl_cfg):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from gen.workloads import CONFIG_NAMES, config

    wl = config(args.config, with_sfa=True, kv_fp8=args.kv_fp8, idx_mx=args.idx_mx)
    cores = oracle_cores()
    n = min(wl.total_q, cores)
    for i in range(args.warmup):
        oracle_step(wl, [(i * n + j) % wl.total_q for j in range(n)])
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_step(wl, [(i * n + j) % wl.total_q for j in range(n)])
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / max(args.steps, 1) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded)",
            "config": {"workload": workload_name(args), "sample_per_step": f"{n} query tokens"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{n} query tokens per step of the {workload_name(args)} workload"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------------------
def measure_prefill_indexer(dev, steps: int, warmup: int, gpu_id: str):
    """The tensor-bound half of the path: the indexer + Top-K of the prefill chunk (4096 new tokens after
    61440 cached ones, 64 x 128 bf16 heads, K = 2048) through dsa_indexer_topk, each call timed with CUDA
    events on its stream, inputs resident.  Algorithmic flops: 2 * Hi * Di per (query, visible position)."""
    import torch

    import sparse_attention_dsa_gb300 as dsa
    from gen.workloads import config

    wl = config(4, with_sfa=False)

    def up(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)

    d = dsa.DsaDims(batch=wl.batch, total_q=wl.total_q, max_q_len=wl.max_q_len, num_pages=wl.num_pages,
                    page_size=wl.page_size, max_pages_per_seq=wl.max_pages_per_seq, idx_heads=wl.idx_heads,
                    idx_dim=wl.idx_dim, idx_dtype=dsa.DSA_BF16, top_k=wl.top_k, attn_heads=128, kv_dim=576,
                    v_dim=512, softmax_scale=wl.softmax_scale, kv_dtype=dsa.DSA_BF16)
    q_idx, w, k_cache = up(wl.q_idx), up(wl.w), up(wl.k_cache)
    pt, sl, cu = up(wl.page_table), up(wl.seq_lens), up(wl.cu_q_lens)
    topk = torch.empty((wl.total_q, wl.top_k), dtype=torch.int32, device=dev)
    ws = torch.zeros((dsa.workspace_size(d) + 3) // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        dsa.indexer_topk(d, q_idx, None, w, k_cache, None, pt, sl, cu, topk, ws, stream)

    for _ in range(max(warmup, 3)):
        call()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_id).start()
    n = max(steps, 5)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    t0 = time.time()
    for i in range(n):
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    # clocks: repeats of the same calls for about half a second around the timed ones
    while time.time() - t0 < 0.5:
        for _ in range(20):
            call()
        torch.cuda.synchronize()
    t1 = time.time()
    sampler.stop()
    if dsa.get_device_error(ws, stream) != 0:
        raise RuntimeError("device error word set in the prefill indexer measurement")
    ms = float(np.median([e[0].elapsed_time(e[1]) for e in ev]))
    flops = indexer_flops(wl)
    tflops = flops / (ms * 1e-3) / 1e12
    _, tc_peak, tc_kind = measured_peaks()
    return {"workload": "prefill_q4096_ctx65536_hi64x128_bf16_k2048", "ms": ms, "achieved": tflops, "unit": "TFLOP/s",
            "peak": tc_peak, "frac": tflops / tc_peak, "algorithmic_flops": flops, "calls": n,
            "peak_source": f"{tc_kind} bf16_tflops (MEASURED_PEAKS.json)" if tc_kind == "measured" else
            "fallback 1900 TF/s",
            "timing": "median of per-call CUDA event pairs on the launching stream, inputs resident (17 MB of keys: "
                      "L2-resident between calls, as in a prefill pass over the chunk's queries)",
            "clocks": sampler.summary(t0, t1)}

def run_ours(args):
    import torch

    import sparse_attention_dsa_gb300 as dsa
    from gen.workloads import CONFIG_NAMES, config

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    dev = torch.device("cuda", local)
    seed = 1000 + args.config + 7919 * rank
    wl = config(args.config, seed=seed, kv_fp8=args.kv_fp8, idx_mx=args.idx_mx)

    def up(a):
        if a is None:
            return None
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            a = a.view(np.int16)
        return torch.from_numpy(a).to(dev)

    d = dsa.DsaDims(batch=wl.batch, total_q=wl.total_q, max_q_len=wl.max_q_len, num_pages=wl.num_pages,
                    page_size=wl.page_size, max_pages_per_seq=wl.max_pages_per_seq, idx_heads=wl.idx_heads,
                    idx_dim=wl.idx_dim,
                    idx_dtype=(dsa.DSA_MXFP8_E4M3 if wl.idx_mx else dsa.DSA_FP8_E4M3) if wl.idx_fp8 else dsa.DSA_BF16,
                    top_k=wl.top_k, attn_heads=wl.attn_heads, kv_dim=wl.kv_dim, v_dim=wl.v_dim,
                    softmax_scale=wl.softmax_scale,
                    kv_dtype=dsa.DSA_FP8_E4M3 if wl.kv_fp8 else dsa.DSA_BF16)
    q_idx, q_scale, w = up(wl.q_idx), up(wl.q_scale), up(wl.w)
    k_cache, k_scale = up(wl.k_cache), up(wl.k_scale)
    q, kv = up(wl.q), up(wl.kv_cache)
    pt, sl, cu = up(wl.page_table), up(wl.seq_lens), up(wl.cu_q_lens)
    T = wl.total_q
    topk = torch.empty((T, wl.top_k), dtype=torch.int32, device=dev)
    out = torch.empty((T, wl.attn_heads, wl.v_dim), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T, wl.attn_heads), dtype=torch.float32, device=dev)
    ws = torch.zeros(dsa.workspace_size(d) // 4, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        # one pass of the hot path through the product call (indexer + Top-K, then sparse attention)
        dsa.fused_decode(d, q_idx, q_scale, w, k_cache, k_scale, q, kv, pt, sl, cu, topk, out, lse, ws, stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if dsa.get_device_error(ws, stream) != 0:
        raise RuntimeError("device error word set during warm-up")

    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    gpu_id = vis.split(",")[local].strip() if vis else str(local)
    sampler = ClockSampler(gpu_id).start()
    # soak: untimed steps so the clock samples see the GPU under this load
    t_soak = time.time()
    while time.time() - t_soak < args.soak_s:
        for _ in range(50):
            step()
        torch.cuda.synchronize()

    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    t_host0 = time.time()
    start.record(stream)
    for i in range(K):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    barrier(dist)
    # clock window: the timed steps are repeated back to back, in blocks of K timed the same way, until the
    # window is long enough for the sampler (every 20 ms) to see the GPU under exactly this load
    block_ms = []
    while time.time() - t_host0 < args.clock_window_s:
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for i in range(K):
            step()
        b1.record(stream)
        torch.cuda.synchronize()
        block_ms.append(b0.elapsed_time(b1) / K)
    t_window1 = time.time()
    # launch durations for the roofline: the same steps with an event pair around each one
    launches_per_step = dsa.fused_decode_launches(d)
    ev_step = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        ev_step[i][0].record(stream)
        step()
        ev_step[i][1].record(stream)
    # per-kernel breakdown: the same work as separate calls with events between them
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for i in range(K):
        ev[i][0].record(stream)
        dsa.indexer_topk(d, q_idx, q_scale, w, k_cache, k_scale, pt, sl, cu, topk, ws, stream)
        ev[i][1].record(stream)
        dsa.sparse_attn(d, q, kv, pt, sl, cu, topk, out, lse, ws, stream)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    # cold L2: every step preceded by a 512 MB write (4x the 129 MB L2), timed with its own event pair
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device=dev)
    ev_cold = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev_cold[i][0].record(stream)
        step()
        ev_cold[i][1].record(stream)
    torch.cuda.synchronize()
    del flush
    sampler.stop()
    total_ms = start.elapsed_time(end)
    cold_ms = sum(e[0].elapsed_time(e[1]) for e in ev_cold) / K
    step_ms = sum(e[0].elapsed_time(e[1]) for e in ev_step) / K
    idx_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    sfa_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    if dsa.get_device_error(ws, stream) != 0:
        raise RuntimeError("device error word set during the timed steps")
    t_max_s = max_over_ranks(dist, total_ms / 1e3)
    tokens = sum_over_ranks(dist, float(T * K))
    value = tokens / t_max_s

    # end to end through the public call with host buffers: every step copies its query-side inputs from
    # pinned host memory, runs the fused call, and copies its outputs (attention output + selection) back
    # to pinned memory.  As a serving loop would, the copies of one step overlap the kernels of its
    # neighbours: inputs and outputs have two device slots, uploads, kernels and downloads run on three
    # streams ordered by events, and the timed region spans the first upload to the last download.
    e2e = None
    if not args.no_e2e:
        host_in = [torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16 else
                                    np.ascontiguousarray(a)).pin_memory()
                   for a in (wl.q_idx, wl.w, wl.q, wl.seq_lens, wl.cu_q_lens, wl.page_table)]
        if wl.idx_fp8:
            host_in.append(torch.from_numpy(np.ascontiguousarray(wl.q_scale)).pin_memory())
        dev_in = [q_idx, w, q, sl, cu, pt] + ([q_scale] if wl.idx_fp8 else [])
        slots = [dict(inp=[torch.empty_like(t) for t in dev_in], topk=torch.empty_like(topk),
                      out=torch.empty_like(out), lse=torch.empty_like(lse), ws=torch.zeros_like(ws),
                      host_out=torch.empty(out.shape, dtype=out.dtype).pin_memory(),
                      host_topk=torch.empty(topk.shape, dtype=topk.dtype).pin_memory(),
                      h2d=torch.cuda.Event(), comp=torch.cuda.Event(), d2h=torch.cuda.Event()) for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = slots[0]["host_out"].numel() * out.element_size() + slots[0]["host_topk"].numel() * topk.element_size()
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        for sl_ in slots:  # every event starts out recorded, so the first waits return at once
            for e in (sl_["comp"], sl_["d2h"]):
                e.record(stream)

        def e2e_step(i):
            sl_ = slots[i % 2]
            inp = sl_["inp"]
            up.wait_event(sl_["comp"])  # the kernels that last read this slot's inputs are done
            with torch.cuda.stream(up):
                for hsrc, dst in zip(host_in, inp):
                    dst.copy_(hsrc, non_blocking=True)
            sl_["h2d"].record(up)
            stream.wait_event(sl_["h2d"])
            stream.wait_event(sl_["d2h"])  # the previous download of this slot's outputs is done
            qi, wi, qq, sli, cui, pti = inp[:6]
            qs = inp[6] if wl.idx_fp8 else q_scale
            dsa.fused_decode(d, qi, qs, wi, k_cache, k_scale, qq, kv, pti, sli, cui, sl_["topk"], sl_["out"],
                             sl_["lse"], sl_["ws"], stream)
            sl_["comp"].record(stream)
            down.wait_event(sl_["comp"])
            with torch.cuda.stream(down):
                sl_["host_out"].copy_(sl_["out"], non_blocking=True)
                sl_["host_topk"].copy_(sl_["topk"], non_blocking=True)
            sl_["d2h"].record(down)

        for i in range(4):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier(dist)
        s2, e2, last = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
                        torch.cuda.Event())
        s2.record(stream)
        up.wait_event(s2)
        for i in range(K):
            e2e_step(i)
        last.record(down)
        stream.wait_event(last)
        e2.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        for sl_ in slots:
            if dsa.get_device_error(sl_["ws"], stream) != 0:
                raise RuntimeError("device error word set during the end-to-end steps")
        if not torch.equal(slots[0]["host_topk"], topk.cpu()):
            raise RuntimeError("end-to-end selection differs from the device-resident run")
        e2e_s = max_over_ranks(dist, s2.elapsed_time(e2) / 1e3)
        e2e = {"value": tokens / e2e_s, "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "overlap": "two device slots; uploads, kernels and downloads of adjacent steps overlap (3 streams)"}

    # roofline of the dominant kernel
    topk_host = topk.cpu().numpy()
    b_idx, b_sfa = indexer_bytes(wl), sfa_bytes(wl, topk_host)
    hbm_peak, _, peak_kind = measured_peaks()
    if launches_per_step == 1:
        # the single-launch kernel carries the whole step
        dominant, alg, dur_ms = "decode", b_idx + b_sfa, step_ms
    else:
        dominant = "indexer" if idx_ms >= sfa_ms else "sfa"
        alg = b_idx if dominant == "indexer" else b_sfa
        dur_ms = idx_ms if dominant == "indexer" else sfa_ms
    achieved = alg / (dur_ms * 1e-3) / 1e9
    traffic = kernel_traffic(dominant, f"{dominant}_{workload_name(args)}.md")
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                "traffic": traffic, "kernel": dominant, "algorithmic_bytes": alg,
                "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured" else
                "fallback 6.8 TB/s"}
    if args.config in TENSOR_BOUND_CONFIGS and not wl.idx_fp8:
        # the indexer's score GEMM dominates: algorithmic bf16 flops over its separate-call duration,
        # against the measured dense bf16 tensor rate
        _, tc_peak, tc_kind = measured_peaks()
        flops = indexer_flops(wl)
        tflops = flops / (idx_ms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "achieved": tflops, "peak": tc_peak, "unit": "TFLOP/s",
                    "frac": tflops / tc_peak, "traffic": kernel_traffic("indexer", f"indexer_{workload_name(args)}.md"),
                    "kernel": "indexer", "algorithmic_flops": flops,
                    "peak_source": f"{tc_kind} bf16_tflops (MEASURED_PEAKS.json)" if tc_kind == "measured" else
                    "fallback 1900 TF/s"}
    step_bytes = b_idx + b_sfa
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": t_max_s * 1e3 / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": (("mxfp8-e4m3 indexer (E8M0 scale per 32)" if wl.idx_mx else "fp8-e4m3 indexer") if wl.idx_fp8
                  else "bf16 indexer") +
        (" / fp8-e4m3 latent-KV cache (128-element tile scales) dequantised to bf16 attention" if wl.kv_fp8 else
         " / bf16 attention") + ", fp32 accumulate",
        "data": "synthetic (seeded SplitMix64; N(0,1) activations, random page table)",
        "config": {"workload": workload_name(args), "batch_per_gpu": wl.batch, "seq_len": int(wl.seq_lens.max()),
                   "query_tokens_per_gpu": T, "top_k": wl.top_k, "idx_heads": wl.idx_heads, "idx_dim": wl.idx_dim,
                   "attn_heads": wl.attn_heads, "kv_dim": wl.kv_dim, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (indexer K cache and latent-KV cache exceed 129 MB); no flush "
                         "in the timed steps; cold_l2 repeats them with a 512 MB flush before each"},
        "kernel_ms": {"step_launch" if launches_per_step == 1 else "step": step_ms,
                      "indexer_separate": idx_ms, "sparse_attn_separate": sfa_ms},
        "launches_per_step": launches_per_step,
        "step_bytes": step_bytes, "step_hbm_frac": step_bytes / (t_max_s / K) / 1e9 / hbm_peak,
        "roofline": roofline, "gpu_launches": launches_per_step * K,
        "clocks": dict(sampler.summary(t_host0, t_window1),
                       window=f"the {K} timed steps and {len(block_ms)} back-to-back repeats of them "
                              f"({t_window1 - t_host0:.2f} s)",
                       repeat_ms_per_step_median=float(np.median(block_ms)) if block_ms else None),
        "cold_l2": {"ms_per_step": cold_ms, "value": T * world / (cold_ms * 1e-3), "unit": UNIT,
                    "hbm_frac": step_bytes / (cold_ms * 1e-3) / 1e9 / hbm_peak,
                    "how": "each step preceded by a 512 MB device write (L2 is 129 MB), per-step CUDA event pairs"},
    }
    if e2e is not None:
        result["e2e"] = e2e
    if not args.no_prefill_indexer and args.config != 4:
        result["prefill_indexer"] = measure_prefill_indexer(dev, K, args.warmup, gpu_id)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl)
        result["cpu_baseline"]["single_thread"] = cpu_single_thread()
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args, args.config)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
