"""Benchmark: fused paged-attention decode v2 on GB300, one JSON line on stdout.

Workload (N=1): Llama-3-8B-shaped single-sequence decode -- B=1, Hq=32, Hkv=8,
D=128, fp16 K/V pools, page_size=16, 32768 tokens of context on a random
permutation of a 4096-page pool; q/K/V ~ N(0,1).  A step is one pass of the
hot path: the partial kernel over every chunk, then the merge kernel (the plan
is built once outside the timed region, as the pages do).  Steps rotate over
three independent input sets (3 x 128 MiB of K/V read between reuses of a set,
more than the 126 MB L2), so every step streams its K/V from HBM.

`value` is decode KV-read GB/s: K+V bytes the step must read (every visible
token, every KV head, both sides) over the device-timed step.  `e2e` repeats
the measurement through the public API with host buffers: every step copies q
and the page table in from pinned host memory, checks the cached plan, runs the
kernels and reads the output and LSE back.

`--impl reference` times the f64 CPU oracle on the host cores instead (a
deliberately slow baseline), on a bounded sample of the same workload.

Multi-GPU: the path shards without any exchange (independent requests / KV
heads), so N ranks run N independent replicas (weak scaling); value is the
sum over ranks of bytes over the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "decode KV-read GB/s (% of GB300 HBM peak) and µs/step at 32K context"
STEP_TWO = "pa_v2_decode_partial + pa_merge_states (merge launched as a programmatic dependent)"
STEP_FUSED = "pa_v2_decode (merge fused into the partial kernel)"
FALLBACK_HBM_GBS = 6800.0
DELAY_CYCLES = 400_000   # device-side delay before the start event (about 200 us at 2 GHz)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sets", type=int, default=3, help="rotating input sets (L2 avoidance)")
    ap.add_argument("--graph", type=int, default=1, help="replay captured CUDA graphs of the steps")
    ap.add_argument("--e2e-steps", type=int, default=5000)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="skip timing the other four workloads")
    ap.add_argument("--context", type=int, default=32768)
    ap.add_argument("--workload", default="llama3_8b_32k",
                    choices=["llama3_8b_32k", "sliding_window_batch", "sparse_token_exact", "cascade_shared_prefix",
                             "tiny_csr", "block_sparse_selection", "crossover", "dsa_sparse_decode"],
                    help="the 32K Llama-3-8B decode is the headline; the others print a per-step line "
                         "(cold L2 for every step)")
    ap.add_argument("--kernel", type=int, default=0,
                    help="plan.kernel: 0 default, 1 CUDA-core partial kernel, 2 (dsa_sparse_decode) the "
                         "warp-level tensor-core second-K-stream kernel")
    ap.add_argument("--tune", action="store_true",
                    help="--workload runs: also time the chunk size picked by the autotuner")
    ap.add_argument("--fused", action="store_true",
                    help="time the one-launch pa_v2_decode (merge fused into the partial kernel) instead of "
                         "pa_v2_decode_partial + pa_merge_states")
    ap.add_argument("--target", type=int, default=0, help="override the plan's CTA target (0: device-derived)")
    ap.add_argument("--chunking", choices=["balanced", "search", "wave-fit", "tuned"], default="balanced",
                    help="headline chunk size: pa_v2_balanced_pages_per_chunk of the plan's own search (same CTA "
                         "count, equal stage counts for the kernel's warps), the search itself, the smallest size "
                         "that fits one wave of the target (pa_v2_wave_fit_pages_per_chunk), or the autotuner's "
                         "pick (autotune.tune, timed launches before the timed region); the search (or, for it, "
                         "the wave fit) is timed beside it")
    ap.add_argument("--pages-per-chunk", type=int, default=0,
                    help="headline: a fixed chunk size instead of --chunking's (the plan's override argument)")
    ap.add_argument("--dsa-batch", default="1,16", help="dsa_sparse_decode: comma-separated batch sizes")
    ap.add_argument("--profile", type=int, default=0,
                    help="profiling mode: run this many eager steps on one input set and exit (no JSON line)")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_over_ranks(ms_total: float, units: float, world: int, device=None):
    """Max of the timed region over ranks and the sum of the units every rank processed.

    With one rank this is the identity.  With several (torch.distributed already initialised), the
    job's time is the slowest rank's and its throughput is all ranks' units over that time."""
    if world <= 1:
        return ms_total, units
    import torch.distributed as dist
    t = torch.tensor([ms_total, units], dtype=torch.float64, device=device)
    mx = t.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(mx[0].item()), float(t[1].item())


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SOURCES = {
    "pa_v2_partial_tc_kernel": ["pa_partial_tc.cu", "pa_partial_tc_body.cuh", "pa_internal.cuh", "pa_device.cuh",
                                "pa_mma.cuh"],
    "pa_v2_partial_tc_two_plan_kernel": ["pa_partial_tc_cascade.cu", "pa_partial_tc_body.cuh", "pa_internal.cuh",
                                         "pa_device.cuh", "pa_mma.cuh"],
    "pa_v2_partial_simt_kernel": ["pa_partial_simt.cu", "pa_internal.cuh", "pa_device.cuh"],
    "pa_v2_partial_extra_tc05_kernel": ["pa_partial_extra_tc05.cu", "pa_internal.cuh", "pa_device.cuh", "pa_mma.cuh"],
}


def kernel_source_hash(kernel: str) -> str:
    """sha256 over the source files that define `kernel` (in KERNEL_SOURCES order)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(ROOT, "paged_attention_decode_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def ncu_traffic(kernel: str, workload: str = "llama3_8b_32k"):
    """Per-launch DRAM bytes (read + write) from the committed ncu summary of `kernel` on `workload`,
    or None when the kernel's sources changed since the capture."""
    path = os.path.join(ROOT, "profiles", f"{kernel.replace('pa_v2_', '')}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_traffic = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    if not m_hash or not m_traffic:
        return None
    return int(m_traffic.group(1)) if kernel_source_hash(kernel) == m_hash.group(1) else None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def mark(self, which):
        setattr(self, which, time.time())

    def summary(self):
        import datetime
        rows = []
        for l in getattr(self, "lines", []):
            p = [x.strip() for x in l.split(",")]
            if len(p) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append({"t": ts, "sm": float(p[1]), "max": float(p[2]), "power": float(p[3]), "hw": p[5],
                             "hwt": p[6], "swt": p[7], "pcap": p[8]})
            except ValueError:
                continue
        t0, t1 = getattr(self, "start", None), getattr(self, "end", None)
        if t0 is not None and t1 is not None:
            rows = [r for r in rows if t0 <= r["t"] <= t1] or rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        load = rows
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                              ("pcap", "sw_power_cap")):
                if r[key] == "Active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


# ---------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------

def oracle_sample(batch, tokens: int):
    """The same workload cut to its first `tokens` tokens: (q, pools, table) for the oracle."""
    import torch as T
    ps = batch.page_size
    pages = -(-tokens // ps)
    lpl = tokens - (pages - 1) * ps
    return (batch.q, batch.k_pool, batch.v_pool, batch.indices[:pages], T.tensor([0, pages], dtype=T.int32),
            T.tensor([lpl], dtype=T.int32), T.tensor([0], dtype=T.int32), batch.scale)


def time_oracle(batch, seconds: float, tokens: int):
    import oracle
    args = oracle_sample(batch, tokens)
    oracle.attention(*oracle_sample(batch, min(tokens, 256)))  # load + warm
    kv_bytes = tokens * batch.num_kv_heads * batch.head_dim * 2 * batch.k_pool.element_size()
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.attention(*args)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return kv_bytes * reps / el / 1e9, reps, el, oracle.num_threads()


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from paged_attention_decode_gb300 import workloads as W
    batch = W.llama3_8b_32k(context=args.context)
    import oracle
    # size one step so that warmup + steps fit in about two minutes
    probe_tokens = 2048
    oracle.attention(*oracle_sample(batch, 64))
    t0 = time.perf_counter()
    oracle.attention(*oracle_sample(batch, probe_tokens))
    per_tok = (time.perf_counter() - t0) / probe_tokens
    budget = 120.0 / max(1, args.steps + args.warmup)
    tokens = int(max(16, min(args.context, budget / max(per_tok, 1e-12))))
    sample = oracle_sample(batch, tokens)
    for _ in range(args.warmup):
        oracle.attention(*sample)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attention(*sample)
    el = time.perf_counter() - t0
    kv_bytes = tokens * batch.num_kv_heads * batch.head_dim * 2 * batch.k_pool.element_size()
    gbs = kv_bytes * args.steps / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "llama3_8b_32k", "batch": 1, "num_qo_heads": 32, "num_kv_heads": 8, "head_dim": 128,
                   "page_size": 16, "context": args.context, "kv_dtype": "f16",
                   "sample_tokens": tokens},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"each step: the first {tokens} of {args.context} context tokens, all 32 heads"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the GPU path
# ---------------------------------------------------------------------------

def run_ours(args):
    world, rank, local = dist_env()
    import numpy as np  # noqa: F401
    from paged_attention_decode_gb300 import build as pa_build
    from paged_attention_decode_gb300 import pa_v2 as pa
    from paged_attention_decode_gb300 import workloads as W

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    pa_build.build()

    # inputs (CPU, seeded) -- rank r uses seeds offset by r so replicas are independent
    if args.profile:
        args.sets, args.no_cpu_baseline = 1, True
    sets_cpu = [W.llama3_8b_32k(seed=1001 + 100 * s + 10000 * rank, context=args.context)
                for s in range(args.sets)]
    b0 = sets_cpu[0]

    # the oracle baseline on rank 0 before any GPU work
    cpu_baseline = None
    if rank == 0 and not args.no_cpu_baseline:
        gbs, reps, el, cores = time_oracle(b0, args.cpu_seconds, args.context)
        cpu_baseline = {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                        "sample": f"the full step ({args.context} tokens x 32 heads) repeated {reps} times "
                                  f"in {el:.1f} s"}

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dt = pa.KV_DTYPES[b0.dtype]
    target = args.target or pa.pa_v2_default_target_ctas(b0.num_qo_heads, b0.num_kv_heads, b0.head_dim,
                                                         b0.page_size, dt)
    plan = pa.pa_v2_plan(b0.indptr, b0.last_page_len, b0.first_page_offset, b0.page_size, b0.num_qo_heads,
                         b0.num_kv_heads, b0.head_dim, dt, target, 0, b0.seq_lens)
    # the search takes the largest size that still reaches the target (113 pages at 32K: 18 chunks of 113
    # and one of 14 per KV head); the kernel's 8 warps take a chunk's 16-row stages in turn, so 113 leaves
    # one warp a 15th stage while 112 gives each 14 with the same CTA count.  The search's size is timed
    # beside the one used (chunking_ab)
    search_ppc = plan.pages_per_chunk
    fit_ppc = pa.pa_v2_wave_fit_pages_per_chunk(b0.indptr, plan.q_groups * plan.num_kv_heads, target)
    alt_ppc = fit_ppc if args.chunking == "search" and not args.pages_per_chunk else search_ppc
    if args.profile and args.chunking == "tuned" and not args.pages_per_chunk:
        raise SystemExit("bench: --profile runs no autotuning; give --pages-per-chunk (or --chunking search)")
    tuned = None
    if args.chunking == "tuned" and not args.pages_per_chunk and not args.profile and args.kernel == 0:
        from paged_attention_decode_gb300 import autotune
        tuned = autotune.tune(b0, dev, target_ctas=target, reps=30, fused=args.fused)
    balanced = pa.pa_v2_balanced_pages_per_chunk(b0.indptr, b0.page_size, search_ppc)
    fixed = args.pages_per_chunk or {"wave-fit": fit_ppc, "balanced": balanced}.get(args.chunking, 0) or (
        tuned.pages_per_chunk if tuned else 0)
    if fixed and fixed != plan.pages_per_chunk:
        plan = pa.pa_v2_plan(b0.indptr, b0.last_page_len, b0.first_page_offset, b0.page_size,
                             b0.num_qo_heads, b0.num_kv_heads, b0.head_dim, dt, target, fixed, b0.seq_lens)
    plan.struct.kernel = args.kernel
    ri, ti, oi = plan.device_arrays(dev)
    sets = [b.to(dev) for b in sets_cpu]
    N, Hq, D, B = plan.num_chunks, b0.num_qo_heads, b0.head_dim, b0.batch
    wv = torch.empty(N, Hq, D, device=dev)
    wl = torch.empty(N, Hq, device=dev)
    out = torch.empty(B, Hq, D, device=dev)
    lse = torch.empty(B, Hq, device=dev)
    stream = torch.cuda.Stream(device=dev)
    kv_bytes = b0.kv_bytes()
    # partial kernel's algorithmic bytes: K/V + q + page ids + chunk arrays + its partial outputs
    partial_bytes = (kv_bytes + b0.q.numel() * 4 + b0.indices.numel() * 4 + N * 8
                     + N * Hq * (D + 1) * 4)

    counters = plan.device_counters(dev)

    def step_two_launch(i):
        d = sets[i % len(sets)]
        pa.pa_v2_decode_partial(plan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len,
                                d.first_page_offset, b0.scale, wv, wl, None, stream, ri, ti)
        if plan.needs_merge:
            pa.pa_merge_states(wv, wl, oi, B, out, lse, None, stream)

    def step_fused(i):
        d = sets[i % len(sets)]
        pa.pa_v2_decode(plan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len, d.first_page_offset,
                        b0.scale, out, lse, (wv, wl), counters, None, stream, ri, ti, oi)

    step = step_fused if args.fused else step_two_launch
    launches_per_step = 1 if args.fused else 1 + int(plan.needs_merge)

    if args.profile:
        with torch.cuda.stream(stream):
            for i in range(args.profile):
                step(i)
        stream.synchronize()
        print(f"profile mode: {args.profile} steps, plan ppc={plan.pages_per_chunk} chunks={N} "
              f"ctas={plan.total_ctas}", flush=True)
        return

    # correctness guard before timing: the arms must agree with the oracle on set 0
    with torch.cuda.stream(stream):
        step(0)
    stream.synchronize()
    import oracle
    ref_o, ref_l = oracle.attention(*oracle_sample(b0, args.context))
    o_now = (out if (plan.needs_merge or args.fused) else wv[:B]).cpu().double().numpy()
    err = float(abs(o_now - ref_o).max())
    if err > 2e-3:
        raise SystemExit(f"bench: GPU output disagrees with the oracle (max|d| = {err:.3e}); refusing to time")

    # The timed steps replay CUDA graphs that hold exactly those steps: one graph of min(K, 600) steps
    # (600 is a multiple of the 3-set rotation, so the rotation continues across replays) replayed
    # K // 600 times, plus one graph of the remaining steps.  Each graph is replayed once untimed after the
    # warm-up steps, so its upload is not timed.
    graphs = []
    G = len(sets) * 10   # steps per graph of the side measurements (partial-only, chunking A/B)
    with torch.cuda.stream(stream):
        for i in range(3):
            step(i)
    stream.synchronize()
    if args.graph:
        per = min(args.steps, 200 * len(sets))
        full, rem = divmod(args.steps, per)
        for n_steps, start, times in ((per, 0, full), (rem, full * per, 1 if rem else 0)):
            if times == 0:
                continue
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n_steps):
                    step(start + i)
            graphs.append((g, n_steps, times))

    def run_steps(k, start=0, timed=False):
        if timed and graphs:
            with torch.cuda.stream(stream):
                for g, _, times in graphs:
                    for _ in range(times):
                        g.replay()
            return
        with torch.cuda.stream(stream):
            for i in range(k):
                step(start + i)

    # Timed region.  nvidia-smi samples clocks from before the warm-up until after the timed steps, so its
    # start-up does not fall between them.  Warm-up: W steps, then one untimed replay of each timed graph
    # (its upload).  After the barrier and synchronisation, a device-side delay queued before the start
    # event (torch.cuda._sleep: the SM spins for DELAY_CYCLES clocks, about 200 us) gives the host time to
    # enqueue the timed graph replays, so the events time the steps back to back on the device rather than
    # the host's enqueue latency.
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        run_steps(args.warmup)
        with torch.cuda.stream(stream):
            for g, _, _ in graphs:
                g.replay()
        stream.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)
        clocks.mark("start")
        with torch.cuda.stream(stream):
            torch.cuda._sleep(DELAY_CYCLES)
        t_start.record(stream)
        run_steps(args.steps, timed=True)
        t_end.record(stream)
        stream.synchronize()
        clocks.mark("end")
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    untimed_graph_steps = sum(n for _, n, _ in graphs)
    ms_total, job_bytes = reduce_over_ranks(t_start.elapsed_time(t_end), float(kv_bytes) * args.steps, world, dev)
    ms_step = ms_total / args.steps

    # per-launch duration of the dominant (partial) kernel: a second timed region replaying a graph of
    # partial launches only (same rotating inputs), CUDA events on the stream the kernel runs on
    def partial_only(i):
        d = sets[i % len(sets)]
        pa.pa_v2_decode_partial(plan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len,
                                d.first_page_offset, b0.scale, wv, wl, None, stream, ri, ti)
    pgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(pgraph, stream=stream):
        for i in range(G):
            partial_only(i)
    reps = max(1, min(args.steps, 20000) // G)
    with torch.cuda.stream(stream):
        for _ in range(3):
            pgraph.replay()
    stream.synchronize()
    p_start = torch.cuda.Event(enable_timing=True)
    p_end = torch.cuda.Event(enable_timing=True)
    p_start.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            pgraph.replay()
    p_end.record(stream)
    stream.synchronize()
    partial_ms = p_start.elapsed_time(p_end) / (reps * G)

    # per-step distribution: one step at a time after a 512 MiB read that evicts L2, CUDA events around
    # each replay of a one-step graph (median and p10-p90 of 200 steps after 10 warm-up steps)
    flush = torch.zeros(128 << 20, dtype=torch.float32, device=dev)
    cold_med, cold_p10, cold_p90 = _time_cold(lambda: step(0), stream, flush, 10, 200, True)
    del flush

    # the chunking choice, measured in this run: the timed step's plan against the other chunking,
    # alternating graph replays of each (same rotating inputs) so that both see the same clocks
    chunking_ab = None
    if alt_ppc and alt_ppc != plan.pages_per_chunk and not args.fused and args.graph:
        chunking_ab = compare_chunkings(args, pa, alt_ppc, sets, b0, dt, target, dev, stream, step, G)
        chunking_ab["alt_chunking"] = "wave-fit" if alt_ppc == fit_ppc and alt_ppc != search_ppc else "search"

    # end to end through the public API with host buffers
    e2e = run_e2e(args, pa, plan, sets_cpu, sets, dev, stream, b0)

    # the other four workloads, each checked against the oracle before it is timed
    per_config = None
    if rank == 0 and not args.no_per_config:
        peak_gbs = measured_peak()[0]
        per_config = {"llama3_8b_32k": {
            "steady": {"us_per_step": ms_step * 1e3, "kv_read_gbs": kv_bytes / (ms_step * 1e-3) / 1e9,
                       "pct_of_hbm_peak": 100.0 * kv_bytes / (ms_step * 1e-3) / 1e9 / peak_gbs,
                       "protocol": "the timed steps above (graph replays, rotating sets)"},
            "cold": {"us_per_step": cold_med, "p10_us": cold_p10, "p90_us": cold_p90,
                     "kv_read_gbs": kv_bytes / (cold_med * 1e-6) / 1e9,
                     "pct_of_hbm_peak": 100.0 * kv_bytes / (cold_med * 1e-6) / 1e9 / peak_gbs,
                     "protocol": "per_step_cold_l2"},
            "kv_bytes_per_step": kv_bytes, "pages_per_chunk": plan.pages_per_chunk, "num_chunks": N,
            "oracle_check": {"max_abs_out": err}}}
        per_config.update(other_configs(args))

    peak, peak_kind = measured_peak()
    timed_protocol = ({"timed_replays": sum(t for _, _, t in graphs),
                       "steps_per_graph": [n for _, n, _ in graphs],
                       "untimed_upload_replay_steps": untimed_graph_steps,
                       "start": f"after a {DELAY_CYCLES}-cycle device-side delay (torch.cuda._sleep) queued after "
                                "the synchronisation, so the replays are enqueued before the start event"}
                      if graphs else False)
    gbs = job_bytes / (ms_total * 1e-3) / 1e9
    achieved = partial_bytes / (partial_ms * 1e-3) / 1e9
    kernel_name = "pa_v2_partial_simt_kernel" if args.kernel == 1 else "pa_v2_partial_tc_kernel"
    traffic = ncu_traffic(kernel_name)
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "us_per_step": ms_step * 1e3,
        "pct_of_hbm_peak": 100.0 * gbs / world / peak, "hbm_peak_gbs": peak, "hbm_peak_kind": peak_kind,
        "pct_of_nominal_8tbs": 100.0 * gbs / world / 8000.0,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": "llama3_8b_32k", "batch": B, "num_qo_heads": Hq, "num_kv_heads": b0.num_kv_heads,
                   "head_dim": D, "page_size": b0.page_size, "context": args.context, "kv_dtype": "f16",
                   "kv_bytes_per_step": kv_bytes, "target_ctas": target, "pages_per_chunk": plan.pages_per_chunk,
                   "chunking": f"fixed {args.pages_per_chunk}" if args.pages_per_chunk else args.chunking,
                   "search_pages_per_chunk": search_ppc, "balanced_pages_per_chunk": balanced,
                   "autotune": None if tuned is None else {
                       "reps": 30, "protocol": "each candidate: median of 30 steps, 512 MiB read before each",
                       "times_us": {str(k): round(v, 2) for k, v in sorted(tuned.times_us.items())}},
                   "wave_fit_pages_per_chunk": fit_ppc,
                   "chunking_ab": chunking_ab,
                   "num_chunks": N, "ctas": plan.total_ctas, "merge": bool(plan.needs_merge),
                   "step": STEP_FUSED if args.fused else STEP_TWO,
                   "l2": f"rotating {len(sets)} independent input sets ({len(sets) * kv_bytes >> 20} MiB of K/V "
                         "between reuses of a set; L2 is 126 MB)",
                   "cuda_graph": timed_protocol, "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm",
                     "kernel": kernel_name, "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": partial_bytes, "launch_us": partial_ms * 1e3,
                     "rest_of_step_us": ms_step * 1e3 - partial_ms * 1e3,
                     "peak_source": f"{peak_kind} hbm_gbs"},
        "per_step_cold_l2": {"median_us": cold_med, "p10_us": cold_p10, "p90_us": cold_p90, "steps": 200,
                             "protocol": "512 MiB read before each step; CUDA events around one graph replay "
                                         "of the step"},
        "per_config": per_config,
        "cpu_baseline": cpu_baseline,
        "e2e": e2e,
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clocks.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


PER_CONFIG = ("tiny_csr", "sliding_window_batch", "sparse_token_exact", "cascade_shared_prefix")


def other_configs(args):
    """us/step and KV-read GB/s of the other four workloads, each arm checked against the oracle first: one
    step at a time after a 512 MiB read (cold L2), median of 100 graph-replayed steps, and (`steady`) steps
    back to back over input variants whose K/V exceeds twice the L2; the cascade workload reports the cascade
    and the flat launch of the same batch."""
    res = {}
    for name in PER_CONFIG:
        ns = argparse.Namespace(**vars(args))
        ns.workload, ns.steps, ns.warmup, ns.tune, ns.profile, ns.graph = name, 100, 10, False, 0, 1
        line = measure_workload(ns)
        arms = line["arms"]
        main = "cascade" if name == "cascade_shared_prefix" else "two"
        peak_gbs = line["hbm_peak_gbs"]
        nbytes = arms[main]["kv_bytes_per_step"]
        entry = {"cold": {"us_per_step": arms[main]["us_per_step_median"], "p10_us": arms[main]["us_p10"],
                          "p90_us": arms[main]["us_p90"], "kv_read_gbs": arms[main]["kv_read_gbs"],
                          "pct_of_hbm_peak": line["pct_of_hbm_peak"],
                          "protocol": "512 MiB read before each step, one graph replay per step, median of 100"},
                 "kv_bytes_per_step": nbytes, "pages_per_chunk": line["config"]["pages_per_chunk"],
                 "num_chunks": line["config"]["num_chunks"], "oracle_check": line["oracle_check"]}
        st = line.get("steady")
        if st:
            entry["steady"] = {"us_per_step": st[main]["us_per_step"], "kv_read_gbs": st[main]["kv_read_gbs"],
                               "pct_of_hbm_peak": 100.0 * st[main]["kv_read_gbs"] / peak_gbs,
                               "fused_us_per_step": st["fused"]["us_per_step"], "variants": st["variants"],
                               "protocol": st["protocol"]}
        if name == "cascade_shared_prefix":
            entry["flat_pages_per_chunk"] = entry.pop("pages_per_chunk")
            entry["flat_num_chunks"] = entry.pop("num_chunks")
            entry["cascade_plan"] = line["config"]["cascade"]
            entry["cold"]["flat_us_per_step"] = arms["two"]["us_per_step_median"]
            entry["cold"]["cascade_over_flat"] = arms["cascade"]["us_per_step_median"] / arms["two"]["us_per_step_median"]
            entry["flat_logical_kv_bytes_per_step"] = arms["two"]["kv_bytes_per_step"]
            if st:
                entry["steady"]["flat_us_per_step"] = st["two"]["us_per_step"]
                entry["steady"]["cascade_over_flat"] = st["cascade"]["us_per_step"] / st["two"]["us_per_step"]
        res[name] = entry
    return res


def compare_chunkings(args, pa, alt_ppc, sets, b0, dt, target, dev, stream, step, G, rounds=5):
    """Median us/step of the timed step's plan and of the plan with `alt_ppc` pages per chunk, from
    `rounds` alternating timed regions of graph replays (two launches per step, as in the timed step)."""
    splan = pa.pa_v2_plan(b0.indptr, b0.last_page_len, b0.first_page_offset, b0.page_size, b0.num_qo_heads,
                          b0.num_kv_heads, b0.head_dim, dt, target, alt_ppc, b0.seq_lens)
    splan.struct.kernel = args.kernel
    sri, sti, soi = splan.device_arrays(dev)
    B, Hq, D = b0.batch, b0.num_qo_heads, b0.head_dim
    swv = torch.empty(splan.num_chunks, Hq, D, device=dev)
    swl = torch.empty(splan.num_chunks, Hq, device=dev)
    sout = torch.empty(B, Hq, D, device=dev)
    slse = torch.empty(B, Hq, device=dev)

    def search_step(i):
        d = sets[i % len(sets)]
        pa.pa_v2_decode_partial(splan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len,
                                d.first_page_offset, b0.scale, swv, swl, None, stream, sri, sti)
        if splan.needs_merge:
            pa.pa_merge_states(swv, swl, soi, B, sout, slse, None, stream)

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(G):
            step(i)
    sgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(sgraph, stream=stream):
        for i in range(G):
            search_step(i)
    reps = max(1, min(args.steps, 20000) // G)

    def timed(g):
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(reps):
                g.replay()
        e.record(stream)
        stream.synchronize()
        return s.elapsed_time(e) * 1e3 / (reps * G)

    ours, search = [], []
    for _ in range(rounds):
        ours.append(timed(graph))
        search.append(timed(sgraph))
    med = lambda v: sorted(v)[len(v) // 2]  # noqa: E731
    return {"us_per_step": med(ours), "alt_us_per_step": med(search), "alt_pages_per_chunk": alt_ppc,
            "alt_ctas": splan.total_ctas, "alt_num_chunks": splan.num_chunks, "rounds": rounds,
            "steps_per_round": reps * G}


def run_e2e(args, pa, plan, sets_cpu, sets, dev, stream, b0):
    """Per step, one call of the C ABI with host buffers: pa_v2_host_graph_run through the binding's
    HostStep on a graph from pa_v2_host_graph_create_mapped -- the cached plan checked against the step's
    page table, the status slot zeroed, one graph launch whose partial kernel reads q and the page table
    from pinned host memory over NVLink-C2C and whose merge writes out and lse2 back into pinned host
    memory -- and the wait for the merge's completion count in the status slot.  Timed beside it: the same step as one direct
    pa_v2_decode_host_mapped call, and both again with copy-engine copies (pa_v2_host_graph_create /
    pa_v2_decode_host: one pinned H2D of the packed inputs into a device buffer, one D2H of the outputs).
    The fused one-launch step (--fused) keeps the per-array path: pa_v2_plan_matches, a pinned copy,
    pa_v2_decode, a copy back."""
    if args.fused:
        return run_e2e_fused(args, pa, plan, sets_cpu, sets, dev, stream, b0)

    def timed(graph, mapped):
        steps = []
        for b, d in zip(sets_cpu, sets):
            st = pa.HostStep(plan, d.k_pool, d.v_pool, stream, graph_scale=b0.scale if graph else None,
                             mapped=mapped)
            st.pack(b.q, b.indices, b.indptr, b.last_page_len, b.first_page_offset)
            steps.append(st)
        for i in range(20):
            steps[i % len(steps)].run(b0.scale)
        n = args.e2e_steps
        t0 = time.perf_counter()
        for i in range(n):
            steps[i % len(steps)].run(b0.scale)
        el = (time.perf_counter() - t0) / n
        o = steps[(n - 1) % len(steps)].out.clone()
        return el, steps[0], o

    copy_direct, _, _ = timed(False, False)
    copy_graph, _, o_copy = timed(True, False)
    mapped_direct, _, _ = timed(False, True)
    per_step, st0, o_mapped = timed(True, True)
    if not torch.equal(o_copy, o_mapped):
        raise RuntimeError("mapped and copied host steps disagree")
    kv_bytes = b0.kv_bytes()
    return {"value": kv_bytes / per_step / 1e9, "unit": "GB/s", "us_per_step": per_step * 1e6,
            "steps": args.e2e_steps, "h2d_bytes_per_step": st0.in_bytes - 16, "d2h_bytes_per_step": st0.out_bytes,
            "direct_call_us_per_step": mapped_direct * 1e6,
            "copy_engine": {"graph_us_per_step": copy_graph * 1e6, "direct_call_us_per_step": copy_direct * 1e6,
                            "h2d_bytes_per_step": st0.in_bytes, "d2h_bytes_per_step": st0.out_bytes},
            "path": "per step: pa_v2_host_graph_run on a pa_v2_host_graph_create_mapped graph (plan check "
                    "against the step's page table, status slot zeroed, one graph launch: " + STEP_TWO +
                    " with q and the page table read by the partial kernel from pinned host memory over "
                    "NVLink-C2C and status + out + lse2 written by the merge into pinned host memory, each merge "
                    "CTA counting itself into the status slot after a system-scope fence; the host waits for "
                    "the full count, then reads the results); direct_call_us_per_step: the same step as one "
                    "pa_v2_decode_host_mapped call; "
                    "copy_engine: the same step with one H2D copy of the packed inputs and one D2H copy of "
                    "the outputs (pa_v2_host_graph_create / pa_v2_decode_host)"}


def run_e2e_fused(args, pa, plan, sets_cpu, sets, dev, stream, b0):
    """The fused step end to end: pa_v2_plan_matches, one pinned H2D of q and the page table,
    pa_v2_decode, one D2H of out + lse, stream sync."""
    B, Hq, D = b0.batch, b0.num_qo_heads, b0.head_dim
    # one pinned staging buffer per input set: [q (f32) | indices | indptr | lpl | fpo] as 32-bit words
    host_in, views = [], []
    for b in sets_cpu:
        parts = [b.q.reshape(-1).view(torch.int32), b.indices, b.indptr, b.last_page_len, b.first_page_offset]
        buf = torch.cat([p.reshape(-1).to(torch.int32) for p in parts]).pin_memory()
        host_in.append((buf, b))
    dev_in = torch.empty(max(h[0].numel() for h in host_in), dtype=torch.int32, device=dev)
    n_q = B * Hq * D
    res_h = torch.empty(B * Hq * (D + 1), dtype=torch.float32).pin_memory()
    res_d = torch.empty(B * Hq * (D + 1), dtype=torch.float32, device=dev)
    out = res_d[:B * Hq * D].view(B, Hq, D)
    lse = res_d[B * Hq * D:].view(B, Hq)
    wv = torch.empty(plan.num_chunks, Hq, D, device=dev)
    wl = torch.empty(plan.num_chunks, Hq, device=dev)
    ri, ti, oi = plan.device_arrays(dev)
    counters = plan.device_counters(dev)
    h2d = host_in[0][0].numel() * 4
    d2h = res_h.numel() * 4

    def one(i):
        buf, b = host_in[i % len(host_in)]
        if not pa.pa_v2_plan_matches(plan, b.indptr, b.last_page_len, b.first_page_offset):
            raise RuntimeError("plan no longer matches")
        nnz = b.indices.numel()
        with torch.cuda.stream(stream):
            dev_in[:buf.numel()].copy_(buf, non_blocking=True)
            q = dev_in[:n_q].view(torch.float32).view(B, Hq, D)
            o = n_q
            idx = dev_in[o:o + nnz]
            o += nnz
            ip = dev_in[o:o + B + 1]
            o += B + 1
            lp = dev_in[o:o + B]
            fp = dev_in[o + B:o + 2 * B]
            kp, vp = sets[i % len(sets)].k_pool, sets[i % len(sets)].v_pool
            pa.pa_v2_decode(plan, q, kp, vp, idx, ip, lp, fp, b0.scale, out, lse, (wv, wl), counters, None,
                            stream, ri, ti, oi)
            res_h.copy_(res_d, non_blocking=True)
        stream.synchronize()

    for i in range(20):
        one(i)
    n = args.e2e_steps
    t0 = time.perf_counter()
    for i in range(n):
        one(i)
    el = time.perf_counter() - t0
    kv_bytes = b0.kv_bytes()
    return {"value": kv_bytes / (el / n) / 1e9, "unit": "GB/s", "us_per_step": el / n * 1e6, "steps": n,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "path": "per step: pa_v2_plan_matches, 1 pinned H2D (q + page table), " + STEP_FUSED
                    + ", 1 D2H (out + lse), stream sync; ctypes binding"}


def run_workload(args):
    line = measure_workload(args)
    if line is not None:
        print(json.dumps(line), flush=True)


def measure_workload(args):
    """Per-step timing of one of the other workloads: every step starts with a cold L2 (a 512 MiB
    buffer is read between steps, outside the event pair).  Arms: "two" = pa_v2_decode_partial +
    pa_merge_states (the default step, `value`), "fused" = the one-launch pa_v2_decode; the cascade adds
    level 0 + level 1 + one pa_merge_states, against the flat arms of the same batch.  The buffer is
    read, not written, so no dirty lines are written back during the step."""
    from paged_attention_decode_gb300 import build as pa_build
    from paged_attention_decode_gb300 import pa_v2 as pa
    from paged_attention_decode_gb300 import workloads as W
    import oracle

    pa_build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.zeros(128 << 20, dtype=torch.float32, device=dev)   # 512 MiB, read between steps
    cascade = args.workload == "cascade_shared_prefix"
    cb = W.cascade_shared_prefix() if cascade else None
    b = cb.flat if cascade else W.WORKLOADS[args.workload]()
    dt = pa.KV_DTYPES[b.dtype]

    def make_plan(indptr, lpl, fpo, hq, seq_lens=None, override=0):
        tgt = pa.pa_v2_default_target_ctas(hq, b.num_kv_heads, b.head_dim, b.page_size, dt)
        return pa.pa_v2_plan(indptr, lpl, fpo, b.page_size, hq, b.num_kv_heads, b.head_dim, dt, tgt, override,
                             seq_lens)

    d = b.to(dev)
    plan = make_plan(b.indptr, b.last_page_len, b.first_page_offset, b.num_qo_heads, b.seq_lens, b.ppc_override)
    search_ppc0 = plan.pages_per_chunk
    chunking = "fixed by the workload" if b.ppc_override else "pa_v2_plan's search"
    wave = pa.pa_v2_default_target_ctas(b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, dt)
    if not b.ppc_override and not cascade and plan.total_ctas > wave:
        # the search's chunk size spills past one wave: take the smallest size that fits it
        fit = pa.pa_v2_wave_fit_pages_per_chunk(b.indptr, plan.q_groups * plan.num_kv_heads, wave)
        plan = make_plan(b.indptr, b.last_page_len, b.first_page_offset, b.num_qo_heads, b.seq_lens, fit)
        chunking = "pa_v2_wave_fit_pages_per_chunk (the search's size spilled past one wave)"
    search_plan = None
    if not b.ppc_override and not cascade and not args.tune and plan.total_ctas <= wave:
        # the largest size at or below the search's with its chunk count that gives the kernel's 8 warps
        # equal stage counts; the search's own plan is timed beside it ("two_search")
        bal = pa.pa_v2_balanced_pages_per_chunk(b.indptr, b.page_size, plan.pages_per_chunk)
        if bal != plan.pages_per_chunk:
            search_plan = plan
            plan = make_plan(b.indptr, b.last_page_len, b.first_page_offset, b.num_qo_heads, b.seq_lens, bal)
            chunking = "pa_v2_balanced_pages_per_chunk of the search's size (equal stage counts per warp)"
    tuned = None
    if args.tune and not cascade:
        from paged_attention_decode_gb300 import autotune
        tuned = autotune.tune(b, dev, reps=20, stream=stream)
        if tuned.pages_per_chunk != plan.pages_per_chunk:
            plan = make_plan(b.indptr, b.last_page_len, b.first_page_offset, b.num_qo_heads, b.seq_lens,
                             tuned.pages_per_chunk)
        chunking = "autotuned"
    out = torch.empty(b.batch, b.num_qo_heads, b.head_dim, device=dev)
    lse = torch.empty(b.batch, b.num_qo_heads, device=dev)

    def workspace(pl):
        return (torch.empty(max(1, pl.num_chunks), pl.num_qo_heads, pl.head_dim, device=dev),
                torch.empty(max(1, pl.num_chunks), pl.num_qo_heads, device=dev))

    ws = workspace(plan)
    o_indptr = plan.device_arrays(dev)[2]

    def flat_step():
        pa.pa_v2_decode(plan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len, d.first_page_offset,
                        b.scale, out, lse, ws, None, None, stream)

    def two_step():
        if plan.needs_merge:
            pa.pa_v2_decode_partial(plan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len,
                                    d.first_page_offset, b.scale, ws[0], ws[1], None, stream)
            pa.pa_merge_states(ws[0], ws[1], o_indptr, b.batch, out, lse, None, stream)
        else:
            pa.pa_v2_decode_partial(plan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len,
                                    d.first_page_offset, b.scale, out, lse, None, stream)

    steps = {"two": (two_step, b.kv_bytes()), "fused": (flat_step, b.kv_bytes())}
    if search_plan is not None:
        s_ws = workspace(search_plan)
        s_oi = search_plan.device_arrays(dev)[2]
        s_out = torch.empty_like(out)
        s_lse = torch.empty_like(lse)

        def two_search_step():
            pa.pa_v2_decode_partial(search_plan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len,
                                    d.first_page_offset, b.scale, s_ws[0], s_ws[1], None, stream)
            pa.pa_merge_states(s_ws[0], s_ws[1], s_oi, b.batch, s_out, s_lse, None, stream)

        steps["two_search"] = (two_search_step, b.kv_bytes())
    if cascade:
        from paged_attention_decode_gb300 import cascade as C
        M, Hq, D = b.q.shape
        Hkv, G = b.num_kv_heads, Hq // b.num_kv_heads
        npre = len(cb.prefix_indices)
        fp1 = torch.zeros(M, dtype=torch.int32)
        cplan = C.cascade_plan(npre, cb.suffix_indptr, cb.suffix_last_page_len, fp1, b.page_size, Hq, Hkv, D, dt,
                               0, cb.suffix_lens)
        c_args = (d.q, d.k_pool, d.v_pool, cb.prefix_indices.to(dev), cb.suffix_indices.to(dev),
                  cb.suffix_indptr.to(dev), cb.suffix_last_page_len.to(dev), fp1.to(dev), b.scale)
        c_out = torch.empty(M, Hq, D, device=dev)
        c_lse = torch.empty(M, Hq, device=dev)

        def cascade_step():
            # level 0 (stacked heads, read in place) and level 1 in one launch, then one merge
            C.cascade_decode(cplan, *c_args, out=c_out, lse2_out=c_lse, stream=stream)

        cas_bytes = (npre * b.page_size + sum(cb.suffix_lens)) * Hkv * D * 2 * b.k_pool.element_size()
        steps["cascade"] = (cascade_step, cas_bytes)

    if args.profile:
        with torch.cuda.stream(stream):
            for _ in range(args.profile):
                for fn, _ in steps.values():
                    fn()
        stream.synchronize()
        print(f"profile mode: {args.workload}, {args.profile} steps of {list(steps)}", flush=True)
        return None

    # correctness guard before timing: every arm against the f64 oracle (max |out - oracle|, and
    # max |lse2 - oracle| where the arm writes the final lse2)
    ref_o, ref_l = oracle.attention(b.q, b.k_pool, b.v_pool, b.indices, b.indptr, b.last_page_len,
                                    b.first_page_offset, b.scale)
    oracle_check = {}

    def check(name, o_t, l_t):
        with torch.cuda.stream(stream):
            o_t.fill_(float("nan"))
            l_t.fill_(float("nan"))
            steps[name][0]()
        stream.synchronize()
        err = float(abs(o_t.cpu().double().numpy() - ref_o).max())
        lg, lr = l_t.cpu().double().numpy(), ref_l
        fin = lr > -float("inf")
        lerr = float(abs(lg[fin] - lr[fin]).max()) if fin.any() else 0.0
        if not (err <= 2e-3 and lerr <= 1e-3 and bool(((lg > -float("inf")) == fin).all())):
            raise SystemExit(f"bench: {name} output disagrees with the oracle ({err:.3e}, lse2 {lerr:.3e}); "
                             "refusing to time")
        oracle_check[name] = {"max_abs_out": err, "max_abs_lse2": lerr}

    check("two", out, lse)
    check("fused", out, lse)
    if search_plan is not None:
        check("two_search", s_out, s_lse)
    if cascade:
        check("cascade", c_out, c_lse)

    res = {}
    for name, (fn, nbytes) in steps.items():
        # each step is replayed from a CUDA graph of that step alone, so the host enqueues it with one call
        # while the flush runs; the events bracket the replay on the launching stream
        run = fn
        if args.graph:
            with torch.cuda.stream(stream):
                for _ in range(3):
                    fn()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            run = g.replay
        times = []
        with torch.cuda.stream(stream):
            for i in range(args.warmup + args.steps):
                flush.sum()   # reads 512 MiB: the next step starts with a cold, clean L2
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                run()
                e1.record(stream)
                times.append((e0, e1))
        stream.synchronize()
        t = sorted(a.elapsed_time(z) for a, z in times[args.warmup:])
        med = t[len(t) // 2]
        res[name] = {"us_per_step_median": med * 1e3, "us_p10": t[len(t) // 10] * 1e3,
                     "us_p90": t[(9 * len(t)) // 10] * 1e3, "kv_bytes_per_step": nbytes,
                     "kv_read_gbs": nbytes / (med * 1e-3) / 1e9}
    steady = None
    if args.workload != "tiny_csr":
        steady = _steady(pa, b, cb, plan, d, dev, stream, cas_bytes if cascade else None,
                         cplan if cascade else None)
    peak, peak_kind = measured_peak()
    main = res["cascade" if cascade else "two"]
    line = {"metric": "decode step us/step (median, cold L2) and KV-read GB/s", "value": main["us_per_step_median"],
            "unit": "us/step", "higher_is_better": False, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "dtype": {"float16": "f16", "bfloat16": "bf16", "float32": "f32"}[str(b.dtype).replace("torch.", "")], "data": "synthetic",
            "config": {"workload": args.workload, "batch": b.batch, "num_qo_heads": b.num_qo_heads,
                       "num_kv_heads": b.num_kv_heads, "head_dim": b.head_dim, "page_size": b.page_size,
                       "kv_dtype": str(b.dtype).replace("torch.", ""), "seq_lens_total": sum(b.seq_lens),
                       "num_chunks": plan.num_chunks, "pages_per_chunk": plan.pages_per_chunk,
                       "chunking": chunking,
                       "search_pages_per_chunk": search_ppc0,
                       "l2": "512 MiB buffer read between steps", "cuda_graph": bool(args.graph)},
            "arms": res, "pct_of_hbm_peak": 100.0 * main["kv_read_gbs"] / peak, "hbm_peak_gbs": peak,
            "steady": steady, "oracle_check": oracle_check}
    if cascade:
        line["config"]["cascade"] = {"level0_pages_per_chunk": cplan.level0.pages_per_chunk,
                                     "level1_pages_per_chunk": cplan.level1.pages_per_chunk,
                                     "level0_chunks": cplan.level0.num_chunks, "level1_chunks": cplan.level1.num_chunks,
                                     "ctas": cplan.level0.total_ctas + cplan.level1.total_ctas,
                                     "merge_rows": cplan.plans.merge_rows}
    if tuned is not None:
        line["autotune"] = {"pages_per_chunk": tuned.pages_per_chunk, "default": tuned.default_pages_per_chunk,
                            "times_us": {str(k): round(v, 2) for k, v in tuned.times_us.items()},
                            "num_chunks": {str(k): v for k, v in tuned.num_chunks.items()}}
    return line


L2_BYTES = 126 << 20


def _steady(pa, b, cb, plan, d, dev, stream, cas_bytes=None, cplan=None, reps=5):
    """Steady-state steps: the step back to back, as a serving loop runs it, over variants of the input whose
    K/V does not repeat within twice the L2 (each variant reads other memory: its page ids point into its own
    copy of the pools, or, for the one-row pages of the sparse workload, at other rows of the same pool), from
    a CUDA graph of several rotations; programmatic dependent launches let each step's kernels start while the
    previous one finishes.  Returns per-step us and KV-read GB/s per arm ("two": partial + merge; "fused": the
    one-launch pa_v2_decode; "cascade")."""
    from paged_attention_decode_gb300 import cascade as C
    unique = cas_bytes if cas_bytes is not None else b.kv_bytes()
    nsets = max(3, min(32, -(-2 * L2_BYTES // unique)))
    P = b.k_pool.shape[0]
    sparse = b.page_size == 1 and b.meta.get("cap")
    if sparse:
        cap = int(b.meta["cap"])
        kp, vp = d.k_pool, d.v_pool
        base = (d.indices // cap) * cap
        pos = d.indices - base
        idx = [base + (pos + 7919 * v) % cap for v in range(nsets)]
    else:
        kp = torch.cat([d.k_pool] * nsets)
        vp = torch.cat([d.v_pool] * nsets)
        idx = [d.indices + v * P for v in range(nsets)]
    ri, ti, oi = plan.device_arrays(dev)
    wv = torch.empty(max(1, plan.num_chunks), plan.num_qo_heads, plan.head_dim, device=dev)
    wl = torch.empty(max(1, plan.num_chunks), plan.num_qo_heads, device=dev)
    out = torch.empty(b.batch, b.num_qo_heads, b.head_dim, device=dev)
    lse = torch.empty(b.batch, b.num_qo_heads, device=dev)

    def two(v):
        if plan.needs_merge:
            pa.pa_v2_decode_partial(plan, d.q, kp, vp, idx[v], d.indptr, d.last_page_len, d.first_page_offset,
                                    b.scale, wv, wl, None, stream, ri, ti)
            pa.pa_merge_states(wv, wl, oi, b.batch, out, lse, None, stream)
        else:
            pa.pa_v2_decode_partial(plan, d.q, kp, vp, idx[v], d.indptr, d.last_page_len, d.first_page_offset,
                                    b.scale, out, lse, None, stream, ri, ti)

    counters = plan.device_counters(dev)

    def fused(v):
        pa.pa_v2_decode(plan, d.q, kp, vp, idx[v], d.indptr, d.last_page_len, d.first_page_offset, b.scale, out, lse,
                        (wv, wl), counters, None, stream, ri, ti, oi)

    arms = {"two": (two, b.kv_bytes()), "fused": (fused, b.kv_bytes())}
    if cplan is not None:
        pre = [cb.prefix_indices.to(dev) + v * P for v in range(nsets)]
        suf = [cb.suffix_indices.to(dev) + v * P for v in range(nsets)]
        sip, slp = cb.suffix_indptr.to(dev), cb.suffix_last_page_len.to(dev)
        sfp = torch.zeros(len(cb.suffix_lens), dtype=torch.int32, device=dev)
        c_out, c_lse = torch.empty_like(out), torch.empty_like(lse)

        def casc(v):
            C.cascade_decode(cplan, d.q, kp, vp, pre[v], suf[v], sip, slp, sfp, b.scale, out=c_out, lse2_out=c_lse,
                             stream=stream)

        arms["cascade"] = (casc, cas_bytes)
    G = nsets * max(1, 60 // nsets)
    res = {"variants": nsets, "steps_per_graph": G, "replays": reps,
           "protocol": "back-to-back graph replays rotating over input variants whose K/V exceeds twice the L2"}
    for name, (fn, nbytes) in arms.items():
        with torch.cuda.stream(stream):
            for v in range(nsets):
                fn(v)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(G):
                fn(i % nsets)
        with torch.cuda.stream(stream):
            g.replay()
            g.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(DELAY_CYCLES)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        stream.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (reps * G)
        res[name] = {"us_per_step": us, "kv_bytes_per_step": nbytes, "kv_read_gbs": nbytes / (us * 1e-6) / 1e9}
    del kp, vp
    return res


def _time_cold(fn, stream, flush, warmup, steps, graph):
    """Median, p10, p90 (us) of `fn` per step with a 512 MiB read before each step, replayed from a CUDA
    graph of that step when `graph`."""
    run = fn
    if graph:
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        run = g.replay
    times = []
    with torch.cuda.stream(stream):
        for _ in range(warmup + steps):
            flush.sum()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run()
            e1.record(stream)
            times.append((e0, e1))
    stream.synchronize()
    t = sorted(a.elapsed_time(z) * 1e3 for a, z in times[warmup:])
    return t[len(t) // 2], t[len(t) // 10], t[(9 * len(t)) // 10]


def run_block_sparse(args):
    """Block-sparse decode (sparse-paged-decode.md): MiniMax-M3 geometry, 16 selected blocks of 128 rows
    plus the partial final block per request.  Arms: "token_exact" = pa_selection_from_blocks + the
    page_size-1 decode (partial + merge), the expansion inside every step; "block_granular" = the same
    selection as 128-row pages of a pool-backed view of the same allocation (page list built once)."""
    from paged_attention_decode_gb300 import build as pa_build
    from paged_attention_decode_gb300 import pa_v2 as pa
    from paged_attention_decode_gb300 import workloads as W
    import oracle

    pa_build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.zeros(128 << 20, dtype=torch.float32, device=dev)
    s = W.block_sparse_selection()
    d = s.to(dev)
    R, n_rep, D = s.q.shape
    C, topk = s.block_size, s.block_ids.shape[1]
    dt = pa.KV_DTYPES[s.k_pool.dtype]
    per = pa.pa_selection_rows_per_request(topk, C, s.kv_len)
    ip, lp, fp = pa.pa_sparse_csr(R, per)
    plan = pa.pa_v2_plan(ip, lp, fp, 1, n_rep, 1, D, dt, pa.pa_v2_default_target_ctas(n_rep, 1, D, 1, dt))
    ipd, lpd, fpd = ip.to(dev), lp.to(dev), fp.to(dev)
    rows = torch.empty(R * per, dtype=torch.int32, device=dev)
    out = torch.empty(R, n_rep, D, device=dev)
    lse = torch.empty(R, n_rep, device=dev)
    ws = (torch.empty(max(1, plan.num_chunks), n_rep, D, device=dev),
          torch.empty(max(1, plan.num_chunks), n_rep, device=dev))

    def token_exact():
        pa.pa_selection_from_blocks(d.block_ids, C, s.kv_len, s.cap, rows, None, stream)
        pa.decode(plan, d.q, d.k_pool, d.v_pool, rows, ipd, lpd, fpd, s.scale, out, lse, ws, None, stream)

    # block-granular page list of the pool view [R * cap / C, C, 1, D]: request r's selected blocks, then
    # its final block (host marshalling of the selection, once)
    bpr = s.cap // C
    nb = -(-s.kv_len // C)
    pages = torch.cat([torch.cat([r * bpr + s.block_ids[r], torch.tensor([r * bpr + nb - 1], dtype=torch.int32)])
                       for r in range(R)]).to(torch.int32)
    ip2 = torch.arange(0, (R + 1) * (topk + 1), topk + 1, dtype=torch.int32)
    lp2 = torch.full((R,), s.kv_len - (nb - 1) * C, dtype=torch.int32)
    fp2 = torch.zeros(R, dtype=torch.int32)
    plan2 = pa.pa_v2_plan(ip2, lp2, fp2, C, n_rep, 1, D, dt, pa.pa_v2_default_target_ctas(n_rep, 1, D, C, dt))
    kp2, vp2 = d.k_pool.reshape(R * bpr, C, 1, D), d.v_pool.reshape(R * bpr, C, 1, D)
    pages_d, ip2d, lp2d, fp2d = pages.to(dev), ip2.to(dev), lp2.to(dev), fp2.to(dev)
    out2 = torch.empty(R, n_rep, D, device=dev)
    lse2 = torch.empty(R, n_rep, device=dev)
    ws2 = (torch.empty(max(1, plan2.num_chunks), n_rep, D, device=dev),
           torch.empty(max(1, plan2.num_chunks), n_rep, device=dev))

    def block_granular():
        pa.decode(plan2, d.q, kp2, vp2, pages_d, ip2d, lp2d, fp2d, s.scale, out2, lse2, ws2, None, stream)

    if args.profile:
        with torch.cuda.stream(stream):
            for _ in range(args.profile):
                token_exact()
                block_granular()
        stream.synchronize()
        print(f"profile mode: block_sparse_selection, {args.profile} steps of [token_exact, block_granular]",
              flush=True)
        return

    # correctness guard against the oracle before timing
    ref_rows, _ = oracle.selection_rows_ref(s.block_ids, C, s.kv_len, s.cap)
    ref_o, _ = oracle.attention(s.q, s.k_pool, s.v_pool, ref_rows, ip, lp, fp, s.scale)
    with torch.cuda.stream(stream):
        token_exact()
        block_granular()
    stream.synchronize()
    if not torch.equal(rows.cpu(), ref_rows):
        raise SystemExit("bench: expanded rows disagree with the oracle; refusing to time")
    for name, got in (("token_exact", out), ("block_granular", out2)):
        err = float(abs(got.cpu().double().numpy() - ref_o).max())
        if not err <= 2e-3:
            raise SystemExit(f"bench: {name} output disagrees with the oracle ({err:.3e}); refusing to time")

    nbytes = R * per * D * 2 * s.k_pool.element_size()
    res = {}
    for name, fn in (("token_exact", token_exact), ("block_granular", block_granular)):
        med, p10, p90 = _time_cold(fn, stream, flush, args.warmup, args.steps, args.graph)
        res[name] = {"us_per_step_median": med, "us_p10": p10, "us_p90": p90, "kv_bytes_per_step": nbytes,
                     "kv_read_gbs": nbytes / (med * 1e-6) / 1e9}
    peak, _ = measured_peak()
    main_arm = res["token_exact"]
    line = {"metric": "decode step us/step (median, cold L2) and KV-read GB/s", "value": main_arm["us_per_step_median"],
            "unit": "us/step", "higher_is_better": False, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "dtype": "f16", "data": "synthetic",
            "config": {"workload": "block_sparse_selection", "requests": R, "num_qo_heads_per_request": n_rep,
                       "head_dim": D, "block_size": C, "topk_blocks": topk, "kv_len": s.kv_len, "cap": s.cap,
                       "rows_per_request": per, "kv_dtype": "float16", "l2": "512 MiB buffer read between steps",
                       "cuda_graph": bool(args.graph), "token_exact_chunks": plan.num_chunks,
                       "block_granular_chunks": plan2.num_chunks},
            "arms": res, "pct_of_hbm_peak": 100.0 * main_arm["kv_read_gbs"] / peak, "hbm_peak_gbs": peak}
    print(json.dumps(line), flush=True)


def run_crossover(args):
    """The pages' performance sweep on GB300 (PR #984, the M1 Ultra validation report; issue #898,
    Performance validation): batch {1, 4, 8} x context {1024, 4096, 16384, 32768}, Llama-3-8B heads
    (Hq 32, Hkv 8, D 128), fp16 pools, page_size 16, random physical pages.  Arms per cell, each a
    CUDA graph of one step after a 512 MiB L2 flush, median of `--steps`:
      v2           this library's decode (pa_v2_decode_partial + pa_merge_states)
      gather_sdpa  gather the pages into contiguous [B, Hkv, ctx, D] K and V (torch index_select), then
                   torch's scaled_dot_product_attention (the pages' gather-then-SDPA path)
      contiguous   scaled_dot_product_attention on K and V already contiguous (the lower bound of the
                   gather path: no gather)
    The query reaches each arm in the form it consumes (f32 for v2, fp16 for SDPA), cast outside the
    timed region."""
    from paged_attention_decode_gb300 import build as pa_build
    from paged_attention_decode_gb300 import pa_v2 as pa
    from paged_attention_decode_gb300 import workloads as W

    pa_build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.zeros(128 << 20, dtype=torch.float32, device=dev)
    F = torch.nn.functional
    Hq, Hkv, D, ps = 32, 8, 128, 16
    cells = []
    for B in (1, 4, 8):
        for ctx in (1024, 4096, 16384, 32768):
            b = W.make_batch(f"crossover_b{B}_c{ctx}", [ctx] * B, [0] * B, ps, Hq, Hkv, D, torch.float16,
                             seed=1100 + B * 7 + ctx // 1024)
            d = b.to(dev)
            dt = pa.KV_DTYPES[b.dtype]
            wave = pa.pa_v2_default_target_ctas(Hq, Hkv, D, ps, dt)
            plan = pa.pa_v2_plan(b.indptr, b.last_page_len, b.first_page_offset, ps, Hq, Hkv, D, dt, wave, 0,
                                 b.seq_lens)
            search_ppc = plan.pages_per_chunk
            if plan.total_ctas > wave:  # the search's size spills past one wave: the size that fits it
                fit = pa.pa_v2_wave_fit_pages_per_chunk(b.indptr, plan.q_groups * plan.num_kv_heads, wave)
                plan = pa.pa_v2_plan(b.indptr, b.last_page_len, b.first_page_offset, ps, Hq, Hkv, D, dt, wave, fit,
                                     b.seq_lens)
            out = torch.empty(B, Hq, D, device=dev)
            lse = torch.empty(B, Hq, device=dev)
            ws = (torch.empty(max(1, plan.num_chunks), Hq, D, device=dev),
                  torch.empty(max(1, plan.num_chunks), Hq, device=dev))
            pages = ctx // ps
            idx = d.indices.view(B, pages).long()
            q16 = d.q.to(torch.float16).view(B, Hq, 1, D)
            kc = d.k_pool[idx].reshape(B, pages * ps, Hkv, D).transpose(1, 2).contiguous()
            vc = d.v_pool[idx].reshape(B, pages * ps, Hkv, D).transpose(1, 2).contiguous()

            def v2():
                pa.decode(plan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len,
                          d.first_page_offset, b.scale, out, lse, ws, None, stream)

            def gather_sdpa():
                k = d.k_pool[idx].reshape(B, pages * ps, Hkv, D).transpose(1, 2)
                v = d.v_pool[idx].reshape(B, pages * ps, Hkv, D).transpose(1, 2)
                return F.scaled_dot_product_attention(q16, k, v, scale=b.scale, enable_gqa=True)

            def contiguous():
                return F.scaled_dot_product_attention(q16, kc, vc, scale=b.scale, enable_gqa=True)

            stream.wait_stream(torch.cuda.current_stream())  # q16, kc, vc were built on the default stream
            with torch.cuda.stream(stream):
                v2()
                ref = contiguous()
            stream.synchronize()
            err = float((out - ref.view(B, Hq, D).float()).abs().max())
            if not err <= 2e-2:
                raise SystemExit(f"bench: crossover B={B} ctx={ctx}: v2 and SDPA disagree ({err:.3e})")
            cell = {"batch": B, "context": ctx, "pages_per_chunk": plan.pages_per_chunk,
                    "search_pages_per_chunk": search_ppc, "ctas": plan.total_ctas,
                    "chunks": plan.num_chunks, "merge": bool(plan.needs_merge)}
            for name, fn in (("v2", v2), ("gather_sdpa", gather_sdpa), ("contiguous", contiguous)):
                med, p10, p90 = _time_cold(fn, stream, flush, args.warmup, args.steps, args.graph)
                cell[name + "_us"] = round(med, 2)
            cell["v2_over_gather"] = round(cell["gather_sdpa_us"] / cell["v2_us"], 3)
            cell["v2_over_contiguous"] = round(cell["contiguous_us"] / cell["v2_us"], 3)
            cells.append(cell)
            del b, d, kc, vc
            torch.cuda.empty_cache()
    line = {"metric": "decode us/step by batch and context (median, cold L2): v2 vs gather-then-SDPA vs "
                      "contiguous SDPA", "unit": "us/step", "higher_is_better": False, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "data": "synthetic",
            "config": {"workload": "crossover", "num_qo_heads": Hq, "num_kv_heads": Hkv, "head_dim": D,
                       "page_size": ps, "kv_dtype": "float16", "l2": "512 MiB buffer read between steps",
                       "cuda_graph": bool(args.graph)},
            "cells": cells}
    print(json.dumps(line), flush=True)


def run_dsa(args):
    """DSA-shaped decode with the second K stream (sparse-paged-decode.md, the DSA paragraphs): 128 query
    heads over one latent KV head, latent 512 + rope 64 per row (the K buffer is 640 wide:
    concat(kv_latent, indexer_key)), values = latent rows, 2048 selected rows per request (token-exact,
    page_size 1).  Batch 1 (the pages' single-sequence case) and batch 16.  Each step is
    pa_v2_decode_partial_extra + pa_merge_states from a CUDA graph after a 512 MiB L2 flush."""
    from paged_attention_decode_gb300 import build as pa_build
    from paged_attention_decode_gb300 import pa_v2 as pa
    from paged_attention_decode_gb300 import workloads as W
    import oracle

    pa_build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.zeros(128 << 20, dtype=torch.float32, device=dev)
    cells = []
    for B in [int(v) for v in args.dsa_batch.split(",")]:
        x = W.dsa_sparse_decode(batch=B)
        b = x.batch
        d = x.to(dev)
        db = d.batch
        dt = pa.KV_DTYPES[b.dtype]
        wave = pa.pa_v2_default_target_ctas(b.num_qo_heads, 1, x.dim, 1, dt)
        plan = pa.pa_v2_plan(b.indptr, b.last_page_len, b.first_page_offset, 1, b.num_qo_heads, 1, x.dim, dt,
                             wave, 0, b.seq_lens)
        # the smallest chunk size whose CTAs fit one wave (the binary-search default can spill a few CTAs
        # into a second wave), rounded up to whole 128-row tiles of the tensor-memory kernel (a partial
        # tile costs the MMAs of a full one)
        from paged_attention_decode_gb300 import cascade as C
        per = plan.q_groups * plan.num_kv_heads
        fit = C.fit_pages_per_chunk([int(n) for n in b.seq_lens], per, wave)
        fit = min(-(-fit // 128) * 128, max(int(n) for n in b.seq_lens))
        if fit != plan.pages_per_chunk:
            plan = pa.pa_v2_plan(b.indptr, b.last_page_len, b.first_page_offset, 1, b.num_qo_heads, 1, x.dim, dt,
                                 wave, fit, b.seq_lens)
        plan.struct.kernel = args.kernel
        out = torch.empty(B, b.num_qo_heads, x.dim, device=dev)
        lse = torch.empty(B, b.num_qo_heads, device=dev)
        ws = (torch.empty(max(1, plan.num_chunks), b.num_qo_heads, x.dim, device=dev),
              torch.empty(max(1, plan.num_chunks), b.num_qo_heads, device=dev))

        def step():
            pa.decode_extra(plan, db.q, d.q_extra, db.k_pool, db.v_pool, d.k_extra_pool, db.indices, db.indptr,
                            db.last_page_len, db.first_page_offset, b.scale, out, lse, ws, None, stream)

        if args.profile:
            with torch.cuda.stream(stream):
                for _ in range(args.profile):
                    step()
            stream.synchronize()
            print(f"profile mode: dsa batch {B}, {args.profile} steps, {plan.total_ctas} CTAs", flush=True)
            continue

        with torch.cuda.stream(stream):
            step()
        stream.synchronize()
        r0 = slice(0, 1)
        ref_o, _ = oracle.attention_extra(b.q[r0], x.q_extra[r0], b.k_pool, x.k_extra_pool, b.v_pool, x.dim,
                                          b.indices[:b.seq_lens[0]], b.indptr[:2], b.last_page_len[r0],
                                          b.first_page_offset[r0], b.scale)
        err = float(abs(out[r0].cpu().double().numpy() - ref_o).max())
        if not err <= 2e-3:
            raise SystemExit(f"bench: dsa output disagrees with the oracle ({err:.3e}); refusing to time")
        med, p10, p90 = _time_cold(step, stream, flush, args.warmup, args.steps, args.graph)
        rows = sum(b.seq_lens)
        nbytes = rows * (x.dim + x.q_extra.shape[-1]) * b.k_pool.element_size()
        flops = 2.0 * rows * b.num_qo_heads * (x.dim + x.q_extra.shape[-1] + x.dim)
        cells.append({"batch": B, "selected_rows_per_request": b.seq_lens[0], "chunks": plan.num_chunks,
                      "ctas": plan.total_ctas, "us_per_step_median": med, "us_p10": p10, "us_p90": p90,
                      "kv_bytes_per_step": nbytes, "kv_read_gbs": nbytes / (med * 1e-6) / 1e9,
                      "flops_per_step": flops, "tflops": flops / (med * 1e-6) / 1e12,
                      "gathered_bytes_per_step": nbytes * plan.q_groups,
                      "gathered_gbs": nbytes * plan.q_groups / (med * 1e-6) / 1e9})
        del x, d, db
        torch.cuda.empty_cache()
    if args.profile:
        return
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tpeak, tkind = float(json.load(f)["bf16_tflops"]), "measured bf16_tflops (burst)"
    except Exception:
        tpeak, tkind = 1900.0, "fallback"
    big = cells[-1]
    roofline = {"bound": "tensor", "achieved": big["tflops"], "peak": tpeak, "unit": "TFLOP/s",
                "frac": big["tflops"] / tpeak,
                "traffic": ncu_traffic("pa_v2_partial_extra_tc05_kernel", "dsa_b16")
                if big["batch"] == 16 and args.kernel == 0 else None,
                "cell": f"batch {big['batch']}",
                "peak_source": tkind,
                "note": "useful flops (QK over 576 dims + PV over 512, per head and row) over the step time; "
                        "the MMAs issued are twice that (q and P as hi + lo halves)"}
    line = {"metric": "DSA decode us/step (median, cold L2), KV-read GB/s and TFLOP/s", "unit": "us/step",
            "value": cells[0]["us_per_step_median"], "higher_is_better": False, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "dsa_sparse_decode", "num_qo_heads": 128, "num_kv_heads": 1, "dim": 512,
                       "extra_dim": 64, "row_stride": 640, "kv_dtype": "bfloat16", "page_size": 1,
                       "kernel": ["pa_v2_partial_extra_tc05_kernel", "pa_v2_partial_extra_kernel",
                                  "pa_v2_partial_extra_tc_kernel"][args.kernel] + " + pa_merge_states",
                       "chunking": "smallest pages_per_chunk whose CTAs fit one wave, in whole 128-row tiles",
                       "l2": "512 MiB buffer read between steps", "cuda_graph": bool(args.graph)},
            "cells": cells, "roofline": roofline}
    hpeak, hkind = measured_peak()
    line["roofline_gather"] = {
        "bound": "hbm", "achieved": big["gathered_gbs"], "peak": hpeak, "unit": "GB/s",
        "frac": big["gathered_gbs"] / hpeak, "cell": f"batch {big['batch']}", "peak_source": f"{hkind} hbm_gbs",
        "note": "bytes the CTAs gather (every selected row once per q-group CTA of its chunk) over the step time "
                "against the HBM copy peak; one SM's intake of scattered rows, not DRAM bandwidth, bounds the "
                "kernel"}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "dsa_sparse_decode":
        run_dsa(args)
    elif args.workload == "crossover":
        run_crossover(args)
    elif args.workload == "block_sparse_selection":
        run_block_sparse(args)
    elif args.workload != "llama3_8b_32k":
        run_workload(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
