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


def cascade_plan(shared_pages: int, suffix_indptr, suffix_last_page_len, suffix_first_page_offset,
                 page_size: int, num_qo_heads: int, num_kv_heads: int, head_dim: int, kv_dtype: int,
                 target_ctas_level0: int, target_ctas_level1: int, suffix_seq_lens=None) -> CascadePlan:
    """Plans for both levels.  The shared span is `shared_pages` full pages; the suffix table is host data."""
    M = len(suffix_indptr) - 1
    p0 = pa.pa_v2_plan([0, shared_pages], [page_size if shared_pages else 0], [0], page_size,
                       M * num_qo_heads, num_kv_heads, head_dim, kv_dtype, target_ctas_level0)
    p0.struct.stack_members = M
    p0.struct.out_row_step = 2
    p1 = pa.pa_v2_plan(suffix_indptr, suffix_last_page_len, suffix_first_page_offset, page_size, num_qo_heads,
                       num_kv_heads, head_dim, kv_dtype, target_ctas_level1, 0, suffix_seq_lens)
    p1.struct.out_row_step = 2
    return CascadePlan(p0, p1, M, num_qo_heads, head_dim, shared_pages)


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
    """out [M, Hq, D], lse2 [M, Hq] of the M members: level 0 + level 1 + one merge (three launches)."""
    dev = q.device
    b = _buffers(cp, dev)
    v_in, lse_in = b["v_in"], b["lse_in"]
    pa.pa_v2_decode(cp.level0, q, k_pool, v_pool, shared_indices, b["ip0"], b["lp0"], b["fp0"], sm_scale,
                    v_in[:, 0], lse_in[:, 0], b["ws0"], None, status, stream)
    pa.pa_v2_decode(cp.level1, q, k_pool, v_pool, suffix_indices, suffix_indptr, suffix_last_page_len,
                    suffix_first_page_offset, sm_scale, v_in[:, 1], lse_in[:, 1], b["ws1"], None, status, stream)
    M, H, D = cp.members, cp.num_qo_heads, cp.head_dim
    return pa.pa_merge_states(v_in.view(2 * M, H, D), lse_in.view(2 * M, H), b["o_indptr"], M, out, lse2_out,
                              status, stream)


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


def plan_batch(indptr, indices, last_page_len, first_page_offset, page_size: int, num_qo_heads: int,
               num_kv_heads: int, head_dim: int, kv_dtype: int, min_shared_pages: int = 16, min_members: int = 2,
               target_ctas_level0: int | None = None, target_ctas_level1: int | None = None):
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
    p0 = pa.pa_v2_plan([0, shared], [page_size], [0], page_size, M * num_qo_heads, num_kv_heads, head_dim, kv_dtype,
                       t0)
    p0.struct.stack_members = M
    p1 = pa.pa_v2_plan(sp["l1_indptr"], sp["l1_last_page_len"], sp["l1_first_page_offset"], page_size,
                       num_qo_heads, num_kv_heads, head_dim, kv_dtype, t1)
    return BatchCascadePlan(p0, p1, M, B, num_qo_heads, head_dim, shared, sp)


def decode_batch(cp: BatchCascadePlan, q, k_pool, v_pool, sm_scale: float, out=None, lse2_out=None, status=None,
                 stream=None):
    """out [B, Hq, D], lse2 [B, Hq] of the whole batch: level 0 + level 1 + one merge (three launches)."""
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
    pa.pa_v2_decode(cp.level0, q, k_pool, v_pool, d["l0_indices"], d["ip0"], d["lp0"], d["fp0"], sm_scale,
                    d["v_in"], d["lse_in"], d["ws0"], None, status, stream, member_rows=d["member_rows"],
                    out_rows=d["l0_out_rows"])
    pa.pa_v2_decode(cp.level1, q, k_pool, v_pool, d["l1_indices"], d["l1_indptr"], d["l1_last_page_len"],
                    d["l1_first_page_offset"], sm_scale, d["v_in"], d["lse_in"], d["ws1"], None, status, stream,
                    out_rows=d["l1_out_rows"])
    return pa.pa_merge_states(d["v_in"], d["lse_in"], d["merge_indptr"], cp.batch, out, lse2_out, status, stream)
