"""Chunk-size autotuning by real launches.

PR #984 ("fused paged-attention decode v2 with CSR page table and cross-CTA
split-KV"), What changed 4: the autotuner op enumerates the feasible chunk
sizes -- powers of two inside the plan's own bounds, plus the heuristic so the
default is measurable -- returns the binary-search value as its default tactic,
and its run performs a real launch, so profiling measures the kernels.

Here the candidates also include the wave-aligned sizes: for k = 1, 2, 3 the
largest pages_per_chunk whose CTA count still fits in k waves of the device
(SM count x resident CTAs per SM).  The binary-search default takes the
largest size whose CTA count *reaches* the target, which can overshoot one
wave by up to (requests x KV heads x q-groups - 1) CTAs and so run a nearly
empty second wave; the wave-aligned sizes are the candidates that avoid it.

The sizes just below the default that keep its CTA count are candidates too
(up to 16 of them).  The tensor-core kernel hands a chunk's stages to its
warps in turn and a launch ends with its busiest warp, so a size a few pages
smaller can give every warp the same number of stages: at 32K tokens of
16-token pages the default 113 leaves one warp a fifteenth stage, 112 = 8 x 14
does not, and it measured about 0.5 us faster per step on GB300.

Each candidate is timed as a decode step on the caller's inputs -- by default
``pa_v2_decode_partial`` then ``pa_merge_states`` (``fused=True``: the one-launch
``pa_v2_decode``) -- each step after a read of a buffer larger than L2, CUDA
events on the launching stream, median of `reps`.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from . import pa_v2 as pa


@dataclass
class TuneResult:
    pages_per_chunk: int                  # the fastest candidate
    default_pages_per_chunk: int          # the binary-search plan's choice (default tactic)
    times_us: dict = field(default_factory=dict)   # candidate -> median microseconds
    num_chunks: dict = field(default_factory=dict)

    @property
    def speedup_over_default(self) -> float:
        return self.times_us[self.default_pages_per_chunk] / self.times_us[self.pages_per_chunk]


def _chunks(pages, ppc):
    return int(sum(max(1, -(-int(p) // ppc)) for p in pages))


def candidates(indptr, num_kv_heads: int, q_groups: int, wave_ctas: int, default_ppc: int, lo: int,
               hi: int, same_ctas: int = 16) -> list[int]:
    """Powers of two in [lo, hi], the default, the smallest size fitting 1, 2 and 3 waves, and up to
    `same_ctas` sizes just below the default with the default's CTA count."""
    ip = torch.as_tensor(indptr).tolist()
    pages = [ip[i + 1] - ip[i] for i in range(len(ip) - 1)]
    cand = {default_ppc, lo, hi}
    p = 1
    while p <= hi:
        if p >= lo:
            cand.add(p)
        p *= 2
    per = num_kv_heads * q_groups
    for k in (1, 2, 3):
        # the smallest ppc whose CTA count fits in k waves (chunk count is non-increasing in ppc)
        a, b = lo, hi
        if _chunks(pages, b) * per > k * wave_ctas:
            continue
        while a < b:
            m = (a + b) // 2
            if _chunks(pages, m) * per <= k * wave_ctas:
                b = m
            else:
                a = m + 1
        cand.add(a)
    n_default = _chunks(pages, default_ppc)
    for c in range(default_ppc - 1, max(lo, default_ppc - same_ctas) - 1, -1):
        if _chunks(pages, c) != n_default:
            break
        cand.add(c)
    return sorted(c for c in cand if lo <= c <= hi or c == default_ppc)


def tune(batch, device=None, target_ctas: int | None = None, reps: int = 20, extra: list[int] | None = None,
         stream=None, fused: bool = False) -> TuneResult:
    """Time a decode step on `batch` (a workloads.PagedBatch, CPU or device) for each candidate chunk size."""
    dev = torch.device(device or "cuda")
    d = batch.to(dev)
    dt = pa.KV_DTYPES[batch.dtype]
    wave = pa.pa_v2_default_target_ctas(batch.num_qo_heads, batch.num_kv_heads, batch.head_dim, batch.page_size, dt)
    target = target_ctas or wave
    base = pa.pa_v2_plan(batch.indptr, batch.last_page_len, batch.first_page_offset, batch.page_size,
                         batch.num_qo_heads, batch.num_kv_heads, batch.head_dim, dt, target, 0, batch.seq_lens)
    cand = candidates(batch.indptr, batch.num_kv_heads, base.q_groups, wave, base.pages_per_chunk,
                      base.lo_pages_per_chunk, base.hi_pages_per_chunk)
    for e in extra or []:
        if e not in cand:
            cand.append(e)
    flush = torch.zeros(128 << 20, dtype=torch.float32, device=dev)   # 512 MiB
    stream = stream or torch.cuda.Stream(device=dev)
    out = torch.empty(batch.batch, batch.num_qo_heads, batch.head_dim, device=dev)
    lse = torch.empty(batch.batch, batch.num_qo_heads, device=dev)
    res = TuneResult(base.pages_per_chunk, base.pages_per_chunk)
    for ppc in cand:
        plan = base if ppc == base.pages_per_chunk else pa.pa_v2_plan(
            batch.indptr, batch.last_page_len, batch.first_page_offset, batch.page_size, batch.num_qo_heads,
            batch.num_kv_heads, batch.head_dim, dt, target, ppc, batch.seq_lens)
        ws = (torch.empty(plan.num_chunks, plan.num_qo_heads, plan.head_dim, device=dev),
              torch.empty(plan.num_chunks, plan.num_qo_heads, device=dev))
        oi = plan.device_arrays(dev)[2]
        evs = []
        with torch.cuda.stream(stream):
            for i in range(reps + 3):
                flush.sum()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                if fused:
                    pa.pa_v2_decode(plan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len,
                                    d.first_page_offset, batch.scale, out, lse, ws, None, None, stream)
                elif plan.needs_merge:
                    pa.pa_v2_decode_partial(plan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len,
                                            d.first_page_offset, batch.scale, ws[0], ws[1], None, stream)
                    pa.pa_merge_states(ws[0], ws[1], oi, batch.batch, out, lse, None, stream)
                else:
                    pa.pa_v2_decode_partial(plan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len,
                                            d.first_page_offset, batch.scale, out, lse, None, stream)
                e1.record(stream)
                evs.append((e0, e1))
        stream.synchronize()
        t = sorted(a.elapsed_time(b) * 1e3 for a, b in evs[3:])
        res.times_us[ppc] = t[len(t) // 2]
        res.num_chunks[ppc] = plan.num_chunks
    res.pages_per_chunk = min(res.times_us, key=res.times_us.get)
    return res
