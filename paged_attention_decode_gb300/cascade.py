"""Two-level (cascade) decode of requests that share a whole-page prefix.

cascade-attention.md (issue #903): when M requests share their first pages, the
shared span is attended once for all of them and each request's private suffix
separately, and the two softmax states of every request merge with the same
closed form the split-KV decode uses.  Here that is three launches of the
library and no other kernel:

1. level 0 -- ``pa_v2_decode`` over the shared pages as ONE request whose query
   heads are the M members' heads stacked ``h0 = kv * (M * G) + m * G + g``
   (plan field ``stack_members = M``): the kernel reads q in place from the
   member layout ``[M, Hq, D]`` and writes member m's result to row ``2m`` of
   the merge input (``out_row_step = 2``), so each K/V element of the span is
   read once per KV head instead of M times;
2. level 1 -- ``pa_v2_decode`` over each member's suffix, written to rows
   ``2m + 1``;
3. ``pa_merge_states`` with ``o_indptr = [0, 2, 4, ..., 2M]``.

Levels 0 and 1 read different pages and write different merge rows, so they
need not run one after the other.  By default (``concurrent=True``) the plans
split one wave of CTAs between the two levels in proportion to the K/V bytes
each reads (each level takes the smallest chunk size whose CTAs fit its share)
and the decode launches level 1 on a side stream forked from the caller's
stream, joining it before the merge: the two launches' fixed start-up and drain
overlap instead of adding up.

This module only builds plans and marshals buffers; every step runs in the
library's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import pa_v2 as pa


@dataclass
class CascadePlan:
    level0: pa.Plan
    level1: pa.Plan
    members: int
    num_qo_heads: int
    head_dim: int
    shared_pages: int
    o_indptr: torch.Tensor | None = None
    buffers: dict | None = None
    concurrent: bool = False


def _chunks(pages, ppc):
    return sum(max(1, -(-p // ppc)) for p in pages)


def fit_pages_per_chunk(pages, ctas_per_chunk: int, budget: int) -> int:
    """Smallest chunk size (pages) whose CTA count sum_r max(1, ceil(pages_r / ppc)) * ctas_per_chunk fits in
    `budget`; the one-chunk-per-request size when nothing fits."""
    pages = [int(p) for p in pages]
    hi = max([1] + pages)
    if _chunks(pages, hi) * ctas_per_chunk > budget:
        return hi
    lo = 1
    while lo < hi:
        m = (lo + hi) // 2
        if _chunks(pages, m) * ctas_per_chunk <= budget:
            hi = m
        else:
            lo = m + 1
    return lo


def split_wave(wave: int, bytes0: int, bytes1: int, ctas0: int, ctas1: int) -> tuple[int, int]:
    """CTA budgets of the two levels: one wave split in proportion to the bytes each level reads, each at
    least one chunk's CTAs (`ctas0`, `ctas1`)."""
    b0 = int(round(wave * bytes0 / max(1, bytes0 + bytes1)))
    b0 = min(max(b0, ctas0), max(ctas0, wave - ctas1))
    return b0, max(ctas1, wave - b0)


def _concurrent_overrides(pages0, pages1, num_qo_heads, num_kv_heads, head_dim, page_size, kv_dtype, members):
    """pages_per_chunk overrides for the two levels sharing one wave (see split_wave)."""
    qg0 = -(-members * (num_qo_heads // num_kv_heads) // pa.pa_v2_q_heads_per_cta(
        members * (num_qo_heads // num_kv_heads), head_dim, kv_dtype))
    qg1 = -(-(num_qo_heads // num_kv_heads) // pa.pa_v2_q_heads_per_cta(num_qo_heads // num_kv_heads, head_dim,
                                                                        kv_dtype))
    wave = pa.pa_v2_default_target_ctas(num_qo_heads, num_kv_heads, head_dim, page_size, kv_dtype)
    per0, per1 = num_kv_heads * qg0, num_kv_heads * qg1
    b0, b1 = split_wave(wave, sum(pages0), sum(pages1), per0, per1 * len(pages1))
    return fit_pages_per_chunk(pages0, per0, b0), fit_pages_per_chunk(pages1, per1, b1)


_side_streams: dict = {}


def _side_stream(device) -> torch.cuda.Stream:
    key = str(torch.device(device))
    if key not in _side_streams:
        _side_streams[key] = torch.cuda.Stream(device=device)
    return _side_streams[key]


def _fork(stream, device):
    """(main, side) streams with the side stream ordered after everything queued on main so far."""
    main = stream if stream is not None else torch.cuda.current_stream(device)
    side = _side_stream(device)
    ev = torch.cuda.Event()
    ev.record(main)
    side.wait_event(ev)
    return main, side


def _join(main, side):
    ev = torch.cuda.Event()
    ev.record(side)
    main.wait_event(ev)


def cascade_plan(shared_pages: int, suffix_indptr, suffix_last_page_len, suffix_first_page_offset,
                 page_size: int, num_qo_heads: int, num_kv_heads: int, head_dim: int, kv_dtype: int,
                 target_ctas_level0: int = 0, target_ctas_level1: int = 0, suffix_seq_lens=None,
                 concurrent: bool = True) -> CascadePlan:
    """Plans for both levels.  The shared span is `shared_pages` full pages; the suffix table is host data.

    concurrent: size both levels to share one wave and run them at the same time (the targets are then
    ignored); otherwise each level is planned against its own target (0: the device default)."""
    M = len(suffix_indptr) - 1
    ip = [int(x) for x in torch.as_tensor(suffix_indptr).tolist()]
    o0 = o1 = 0
    if concurrent:
        o0, o1 = _concurrent_overrides([shared_pages], [ip[i + 1] - ip[i] for i in range(M)], num_qo_heads,
                                       num_kv_heads, head_dim, page_size, kv_dtype, M)
    t0 = target_ctas_level0 or pa.pa_v2_default_target_ctas(M * num_qo_heads, num_kv_heads, head_dim, page_size,
                                                            kv_dtype)
    t1 = target_ctas_level1 or pa.pa_v2_default_target_ctas(num_qo_heads, num_kv_heads, head_dim, page_size,
                                                            kv_dtype)
    p0 = pa.pa_v2_plan([0, shared_pages], [page_size if shared_pages else 0], [0], page_size,
                       M * num_qo_heads, num_kv_heads, head_dim, kv_dtype, t0, o0)
    p0.struct.stack_members = M
    p0.struct.out_row_step = 2
    p1 = pa.pa_v2_plan(suffix_indptr, suffix_last_page_len, suffix_first_page_offset, page_size, num_qo_heads,
                       num_kv_heads, head_dim, kv_dtype, t1, o1, suffix_seq_lens)
    p1.struct.out_row_step = 2
    return CascadePlan(p0, p1, M, num_qo_heads, head_dim, shared_pages, concurrent=concurrent)


def _buffers(cp: CascadePlan, device) -> dict:
    if cp.buffers is None or cp.buffers["device"] != str(device):
        M, H, D = cp.members, cp.num_qo_heads, cp.head_dim

        def ws(pl):
            return (torch.empty(max(1, pl.num_chunks), pl.num_qo_heads, pl.head_dim, device=device),
                    torch.empty(max(1, pl.num_chunks), pl.num_qo_heads, device=device))

        cp.buffers = {"device": str(device),
                      "v_in": torch.empty(M, 2, H, D, device=device), "lse_in": torch.empty(M, 2, H, device=device),
                      "o_indptr": torch.arange(0, 2 * M + 1, 2, dtype=torch.int32, device=device),
                      "ws0": ws(cp.level0), "ws1": ws(cp.level1),
                      "ip0": torch.tensor([0, cp.shared_pages], dtype=torch.int32, device=device),
                      "lp0": torch.tensor([cp.level0.page_size], dtype=torch.int32, device=device),
                      "fp0": torch.zeros(1, dtype=torch.int32, device=device)}
    return cp.buffers


def cascade_decode(cp: CascadePlan, q, k_pool, v_pool, shared_indices, suffix_indices, suffix_indptr,
                   suffix_last_page_len, suffix_first_page_offset, sm_scale: float, out=None, lse2_out=None,
                   status=None, stream=None):
    """out [M, Hq, D], lse2 [M, Hq] of the M members: level 0 + level 1 + one merge (three launches; the
    two levels on two streams when the plan is concurrent)."""
    dev = q.device
    b = _buffers(cp, dev)
    v_in, lse_in = b["v_in"], b["lse_in"]
    main, side = _fork(stream, dev) if cp.concurrent else (stream, stream)
    # level 0 first: queued the other way round, the merge after the join started ~10 us later (measured
    # in CUDA graphs on GB300)
    pa.pa_v2_decode(cp.level0, q, k_pool, v_pool, shared_indices, b["ip0"], b["lp0"], b["fp0"], sm_scale,
                    v_in[:, 0], lse_in[:, 0], b["ws0"], None, status, main)
    pa.pa_v2_decode(cp.level1, q, k_pool, v_pool, suffix_indices, suffix_indptr, suffix_last_page_len,
                    suffix_first_page_offset, sm_scale, v_in[:, 1], lse_in[:, 1], b["ws1"], None, status, side)
    if cp.concurrent:
        _join(main, side)
    M, H, D = cp.members, cp.num_qo_heads, cp.head_dim
    return pa.pa_merge_states(v_in.view(2 * M, H, D), lse_in.view(2 * M, H), b["o_indptr"], M, out, lse2_out,
                              status, main)


# ---------------------------------------------------------------------------
# cascade over a flat batch: detection, level split, three launches
# ---------------------------------------------------------------------------

@dataclass
class BatchCascadePlan:
    """A detected cascade over a flat batch (members share `shared_pages` leading pages)."""

    level0: pa.Plan
    level1: pa.Plan
    members: int
    batch: int
    num_qo_heads: int
    head_dim: int
    shared_pages: int
    host: dict
    dev: dict | None = None
    concurrent: bool = False


def plan_batch(indptr, indices, last_page_len, first_page_offset, page_size: int, num_qo_heads: int,
               num_kv_heads: int, head_dim: int, kv_dtype: int, min_shared_pages: int = 16, min_members: int = 2,
               target_ctas_level0: int | None = None, target_ctas_level1: int | None = None,
               concurrent: bool = True):
    """Detect a shared prefix in a flat batch (host arrays) and plan both levels, or None if none qualifies.

    Members (the detected group) get two merge rows -- level 0, then level 1 over the pages after the
    shared span; every other request keeps its whole table at level 1 and merges as a single row."""
    member_of, shared = pa.pa_v2_cascade_detect(indptr, indices, first_page_offset, min_shared_pages, min_members)
    M = int(member_of.sum())
    if M == 0:
        return None
    sp = pa.pa_v2_cascade_split(indptr, indices, last_page_len, first_page_offset, member_of, shared)
    ip = torch.as_tensor(indptr).to(torch.int32)
    first = int(sp["member_rows"][0])
    sp["l0_indices"] = torch.as_tensor(indices).to(torch.int32)[int(ip[first]):int(ip[first]) + shared].clone()
    B = len(ip) - 1
    t0 = target_ctas_level0 or pa.pa_v2_default_target_ctas(M * num_qo_heads, num_kv_heads, head_dim, page_size,
                                                             kv_dtype)
    t1 = target_ctas_level1 or pa.pa_v2_default_target_ctas(num_qo_heads, num_kv_heads, head_dim, page_size,
                                                            kv_dtype)
    o0 = o1 = 0
    if concurrent:
        l1 = [int(x) for x in torch.as_tensor(sp["l1_indptr"]).tolist()]
        o0, o1 = _concurrent_overrides([shared], [l1[i + 1] - l1[i] for i in range(len(l1) - 1)], num_qo_heads,
                                       num_kv_heads, head_dim, page_size, kv_dtype, M)
    p0 = pa.pa_v2_plan([0, shared], [page_size], [0], page_size, M * num_qo_heads, num_kv_heads, head_dim, kv_dtype,
                       t0, o0)
    p0.struct.stack_members = M
    p1 = pa.pa_v2_plan(sp["l1_indptr"], sp["l1_last_page_len"], sp["l1_first_page_offset"], page_size,
                       num_qo_heads, num_kv_heads, head_dim, kv_dtype, t1, o1)
    return BatchCascadePlan(p0, p1, M, B, num_qo_heads, head_dim, shared, sp, concurrent=concurrent)


def decode_batch(cp: BatchCascadePlan, q, k_pool, v_pool, sm_scale: float, out=None, lse2_out=None, status=None,
                 stream=None):
    """out [B, Hq, D], lse2 [B, Hq] of the whole batch: level 0 + level 1 + one merge (three launches; the
    two levels on two streams when the plan is concurrent)."""
    dev = q.device
    if cp.dev is None or cp.dev["device"] != str(dev):
        rows = int(cp.host["merge_indptr"][-1])
        H, D = cp.num_qo_heads, cp.head_dim

        def ws(pl):
            return (torch.empty(max(1, pl.num_chunks), pl.num_qo_heads, pl.head_dim, device=dev),
                    torch.empty(max(1, pl.num_chunks), pl.num_qo_heads, device=dev))

        cp.dev = {"device": str(dev), "v_in": torch.empty(rows, H, D, device=dev),
                  "lse_in": torch.empty(rows, H, device=dev), "ws0": ws(cp.level0), "ws1": ws(cp.level1),
                  "ip0": torch.tensor([0, cp.shared_pages], dtype=torch.int32, device=dev),
                  "lp0": torch.tensor([cp.level0.page_size], dtype=torch.int32, device=dev),
                  "fp0": torch.zeros(1, dtype=torch.int32, device=dev)}
        for k in ("l0_indices", "l1_indptr", "l1_indices", "l1_last_page_len", "l1_first_page_offset",
                  "member_rows", "l0_out_rows", "l1_out_rows", "merge_indptr"):
            cp.dev[k] = cp.host[k].to(dev)
    d = cp.dev
    main, side = _fork(stream, dev) if cp.concurrent else (stream, stream)
    pa.pa_v2_decode(cp.level0, q, k_pool, v_pool, d["l0_indices"], d["ip0"], d["lp0"], d["fp0"], sm_scale,
                    d["v_in"], d["lse_in"], d["ws0"], None, status, main, member_rows=d["member_rows"],
                    out_rows=d["l0_out_rows"])
    pa.pa_v2_decode(cp.level1, q, k_pool, v_pool, d["l1_indices"], d["l1_indptr"], d["l1_last_page_len"],
                    d["l1_first_page_offset"], sm_scale, d["v_in"], d["lse_in"], d["ws1"], None, status, side,
                    out_rows=d["l1_out_rows"])
    if cp.concurrent:
        _join(main, side)
    return pa.pa_merge_states(d["v_in"], d["lse_in"], d["merge_indptr"], cp.batch, out, lse2_out, status, main)
