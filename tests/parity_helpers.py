"""Helpers shared by the GPU parity tests: run the C-ABI path and compare with the oracle.

Tolerances (fp16/bf16/fp32 K/V, f32 accumulation) against the f64 oracle on the
same stored values: max |out - ref| <= 2e-3, max |lse2 - ref| <= 1e-3; -inf LSEs
(empty chunks or rows) must match exactly and their outputs must be exactly 0.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_attention_decode_gb300 import pa_v2 as pa

OUT_TOL = 2e-3
LSE_TOL = 1e-3


def assert_close(out, lse, ref_o, ref_l, what=""):
    o = out.detach().cpu().double().numpy()
    l = lse.detach().cpu().double().numpy()
    assert o.shape == ref_o.shape and l.shape == ref_l.shape, (what, o.shape, ref_o.shape)
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(l), fin), f"{what}: -inf pattern differs"
    assert np.all(l[~fin] == -np.inf), what
    assert np.all(o[~fin] == 0.0), f"{what}: empty rows must be exactly zero"
    err_o = float(np.abs(o - ref_o).max()) if o.size else 0.0
    err_l = float(np.abs(l[fin] - ref_l[fin]).max()) if fin.any() else 0.0
    assert err_o <= OUT_TOL, f"{what}: max|dout| = {err_o:.3e}"
    assert err_l <= LSE_TOL, f"{what}: max|dlse2| = {err_l:.3e}"
    return err_o, err_l


def make_plan(b, target=None, override=None):
    tgt = target if target is not None else pa.pa_v2_default_target_ctas(
        b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, pa.KV_DTYPES[b.dtype])
    ovr = b.ppc_override if override is None else override
    return pa.pa_v2_plan(b.indptr, b.last_page_len, b.first_page_offset, b.page_size, b.num_qo_heads,
                         b.num_kv_heads, b.head_dim, pa.KV_DTYPES[b.dtype], tgt, ovr, b.seq_lens)


def run_gpu(b, plan, d=None):
    """Partial then merge through the C ABI.  Returns (partials, lse_partials, out, lse, status)."""
    d = d if d is not None else b.to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    v, l = pa.pa_v2_decode_partial(plan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len,
                                   d.first_page_offset, b.scale, status=status)
    if plan.needs_merge:
        _, _, oi = plan.device_arrays(v.device)
        o, lo = pa.pa_merge_states(v, l, oi, b.batch, status=status)
    else:
        o, lo = v[:b.batch], l[:b.batch]
    torch.cuda.synchronize()
    return v[:plan.num_chunks], l[:plan.num_chunks], o, lo, int(status.item())


def run_gpu_fused(b, plan, d=None):
    """The one-launch decode (pa_v2_decode), twice in a row on the same counters.  Returns (out, lse, status)."""
    d = d if d is not None else b.to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(2):
        o, lo = pa.pa_v2_decode(plan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len,
                                d.first_page_offset, b.scale, status=status)
        outs.append((o.clone(), lo.clone()))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1]), \
        "fused decode is not repeatable (ticket counters not reset?)"
    if plan.num_chunks:
        assert int(plan.device_counters("cuda").abs().sum()) == 0, "ticket counters left non-zero"
    return outs[0][0], outs[0][1], int(status.item())


def check_batch(b, plan=None, target=None, override=None, check_partials=True, d=None, fused=True):
    plan = plan if plan is not None else make_plan(b, target, override)
    d = d if d is not None else b.to("cuda")
    v, l, o, lo, st = run_gpu(b, plan, d)
    assert st == 0, f"{b.name}: device status {st}"
    ref_o, ref_l = oracle.attention(b.q, b.k_pool, b.v_pool, b.indices, b.indptr, b.last_page_len,
                                    b.first_page_offset, b.scale)
    errs = assert_close(o, lo, ref_o, ref_l, f"{b.name} merged (ppc={plan.pages_per_chunk})")
    if fused:
        fo, fl, fst = run_gpu_fused(b, plan, d)
        assert fst == 0, f"{b.name}: fused device status {fst}"
        assert_close(fo, fl, ref_o, ref_l, f"{b.name} fused (ppc={plan.pages_per_chunk})")
    if check_partials:
        pv, pl = oracle.partials(b.q, b.k_pool, b.v_pool, b.indices, b.indptr, b.last_page_len,
                                 b.first_page_offset, b.scale, plan.pages_per_chunk, plan.request_indices,
                                 plan.kv_tile_indices)
        assert_close(v, l, pv, pl, f"{b.name} partials (ppc={plan.pages_per_chunk})")
    return plan, o, lo, errs
