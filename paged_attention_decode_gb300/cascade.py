"""Two-level (cascade) decode of requests that share a whole-page prefix.

cascade-attention.md (issue #903): when M requests share their first pages, the
shared span is attended once for all of them and each request's private suffix
separately, and the two softmax states of every request merge with the same
closed form the split-KV decode uses.  Here that is two launches of the
library, both from one C call (``pa_v2_cascade_decode``):

1. ONE launch of the partial kernel over both levels' chunks --
   level 0, the shared pages as ONE request whose query heads are the M
   members' heads stacked ``h0 = kv * (M * G) + m * G + g`` (plan field
   ``stack_members = M``; q read in place from the member layout
   ``[M, Hq, D]``), so each K/V element of the span is read once per KV head
   instead of M times; and level 1, each request's own pages.  Every chunk's
   normalized partial lands in one merge input, request by request: a
   member's level-0 chunks, then its level-1 chunks;
2. ``pa_merge_states`` over each request's rows (the merge is associative, so
   folding a request's chunks of both levels at once is the cascade's
   two-state merge).

``pa_v2_cascade_plan`` sizes the chunks so both levels fit one wave and run
side by side: level 1 at the smallest common size whose CTAs over both levels
fit, level 0 (whose chunks carry every member's stacked heads) at the smallest
size that uses the CTAs left over.  For a flat batch, ``pa_v2_cascade_detect``
finds the shared prefix and ``pa_v2_cascade_split`` builds the level-1 table
and the row maps.

This module only builds plans and marshals buffers; every step runs in the
library's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import pa_v2 as pa


@dataclass
class CascadePlan:
    plans: pa.CascadePlans
    members: int
    num_qo_heads: int
    head_dim: int
    shared_pages: int
    buffers: dict | None = None

    @property
    def level0(self) -> pa.Plan:
        return self.plans.level0

    @property
    def level1(self) -> pa.Plan:
        return self.plans.level1


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


def _wave(num_qo_heads, num_kv_heads, head_dim, page_size, kv_dtype):
    return pa.pa_v2_default_target_ctas(num_qo_heads, num_kv_heads, head_dim, page_size, kv_dtype)


def cascade_plan(shared_pages: int, suffix_indptr, suffix_last_page_len, suffix_first_page_offset,
                 page_size: int, num_qo_heads: int, num_kv_heads: int, head_dim: int, kv_dtype: int,
                 wave_ctas: int = 0, suffix_seq_lens=None) -> CascadePlan:
    """Plans for both levels (pa_v2_cascade_plan: chunk sizes whose CTAs fit one wave of `wave_ctas`, 0 =
    the device's).  The shared span is `shared_pages` full pages; the suffix table is host data."""
    M = len(suffix_indptr) - 1
    wave = wave_ctas or _wave(num_qo_heads, num_kv_heads, head_dim, page_size, kv_dtype)
    cps = pa.pa_v2_cascade_plan(M, shared_pages, suffix_indptr, suffix_last_page_len, suffix_first_page_offset,
                                page_size, num_qo_heads, num_kv_heads, head_dim, kv_dtype, wave, suffix_seq_lens)
    return CascadePlan(cps, M, num_qo_heads, head_dim, shared_pages)


def _level_tables(cps: pa.CascadePlans, shared_pages: int, page_size: int, device) -> dict:
    H, D = cps.level1.num_qo_heads, cps.level1.head_dim
    return {"device": str(device),
            "merge_v": torch.empty(cps.merge_rows, H, D, device=device),
            "merge_lse": torch.empty(cps.merge_rows, H, device=device),
            "merge_indptr": cps.merge_indptr.to(device),
            "l0_part_rows": cps.l0_part_rows.to(device), "l1_part_rows": cps.l1_part_rows.to(device),
            "ip0": torch.tensor([0, shared_pages], dtype=torch.int32, device=device),
            "lp0": torch.tensor([page_size], dtype=torch.int32, device=device),
            "fp0": torch.zeros(1, dtype=torch.int32, device=device)}


def cascade_decode(cp: CascadePlan, q, k_pool, v_pool, shared_indices, suffix_indices, suffix_indptr,
                   suffix_last_page_len, suffix_first_page_offset, sm_scale: float, out=None, lse2_out=None,
                   status=None, stream=None):
    """out [M, Hq, D], lse2 [M, Hq] of the M members: both levels in one launch, then one merge."""
    dev = q.device
    if cp.buffers is None or cp.buffers["device"] != str(dev):
        cp.buffers = _level_tables(cp.plans, cp.shared_pages, cp.level0.page_size, dev)
    b = cp.buffers
    lv0 = pa.cascade_level(cp.level0, shared_indices, b["ip0"], b["lp0"], b["fp0"], b["l0_part_rows"])
    lv1 = pa.cascade_level(cp.level1, suffix_indices, suffix_indptr, suffix_last_page_len, suffix_first_page_offset,
                           b["l1_part_rows"])
    return pa.pa_v2_cascade_decode(cp.plans, lv0, lv1, q, k_pool, v_pool, sm_scale, b["merge_v"], b["merge_lse"],
                                   b["merge_indptr"], out, lse2_out, status, stream)


# ---------------------------------------------------------------------------
# cascade over a flat batch: detection, level split, one call
# ---------------------------------------------------------------------------

@dataclass
class BatchCascadePlan:
    """A detected cascade over a flat batch (members share `shared_pages` leading pages)."""

    plans: pa.CascadePlans
    members: int
    batch: int
    num_qo_heads: int
    head_dim: int
    shared_pages: int
    host: dict
    dev: dict | None = None

    @property
    def level0(self) -> pa.Plan:
        return self.plans.level0

    @property
    def level1(self) -> pa.Plan:
        return self.plans.level1


def plan_batch(indptr, indices, last_page_len, first_page_offset, page_size: int, num_qo_heads: int,
               num_kv_heads: int, head_dim: int, kv_dtype: int, min_shared_pages: int = 16, min_members: int = 2,
               wave_ctas: int = 0):
    """Detect a shared prefix in a flat batch (host arrays) and plan both levels, or None if none qualifies.

    Members (the detected group) read the shared span at level 0 and the pages after it at level 1; every
    other request keeps its whole table at level 1."""
    member_of, shared = pa.pa_v2_cascade_detect(indptr, indices, first_page_offset, min_shared_pages, min_members)
    M = int(member_of.sum())
    if M == 0:
        return None
    sp = pa.pa_v2_cascade_split(indptr, indices, last_page_len, first_page_offset, member_of, shared)
    ip = torch.as_tensor(indptr).to(torch.int32)
    first = int(sp["member_rows"][0])
    sp["l0_indices"] = torch.as_tensor(indices).to(torch.int32)[int(ip[first]):int(ip[first]) + shared].clone()
    B = len(ip) - 1
    wave = wave_ctas or _wave(num_qo_heads, num_kv_heads, head_dim, page_size, kv_dtype)
    cps = pa.pa_v2_cascade_plan(M, shared, sp["l1_indptr"], sp["l1_last_page_len"], sp["l1_first_page_offset"],
                                page_size, num_qo_heads, num_kv_heads, head_dim, kv_dtype, wave,
                                member_requests=sp["member_rows"])
    return BatchCascadePlan(cps, M, B, num_qo_heads, head_dim, shared, sp)


def decode_batch(cp: BatchCascadePlan, q, k_pool, v_pool, sm_scale: float, out=None, lse2_out=None, status=None,
                 stream=None):
    """out [B, Hq, D], lse2 [B, Hq] of the whole batch: both levels in one launch, then one merge."""
    dev = q.device
    if cp.dev is None or cp.dev["device"] != str(dev):
        cp.dev = _level_tables(cp.plans, cp.shared_pages, cp.level0.page_size, dev)
        for k in ("l0_indices", "l1_indptr", "l1_indices", "l1_last_page_len", "l1_first_page_offset",
                  "member_rows"):
            cp.dev[k] = cp.host[k].to(dev)
    d = cp.dev
    lv0 = pa.cascade_level(cp.level0, d["l0_indices"], d["ip0"], d["lp0"], d["fp0"], d["l0_part_rows"],
                           member_rows=d["member_rows"])
    lv1 = pa.cascade_level(cp.level1, d["l1_indices"], d["l1_indptr"], d["l1_last_page_len"],
                           d["l1_first_page_offset"], d["l1_part_rows"])
    return pa.pa_v2_cascade_decode(cp.plans, lv0, lv1, q, k_pool, v_pool, sm_scale, d["merge_v"], d["merge_lse"],
                                   d["merge_indptr"], out, lse2_out, status, stream)
