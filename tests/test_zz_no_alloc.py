"""pa_v2_decode_noalloc against the f64 oracle and against pa_v2_decode (GPU).

Some callers cannot allocate device memory -- for example a serving engine that
has reserved the whole GPU for its own pools, or a plugin that its host hands
only input and output pointers -- so they cannot supply the workspace and
ticket counters pa_v2_decode needs.  pa_v2_decode_noalloc takes both from the
library's fixed device array instead.  These tests call it through the C ABI,
twice in a row on the same array, and compare each result with the oracle
(max |out| error 2e-3, max |lse2| error 1e-3) and with pa_v2_decode on the same
inputs; they cover plans that merge, a one-chunk-per-request plan, an empty
batch, a stacked cascade-level plan whose rows land out_row_step apart, and a
plan too large for the array, which is refused before any launch.  The file
sorts last so that a run stopping at the first failure has already run every
other test.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_attention_decode_gb300 import pa_v2 as pa
from paged_attention_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu

OUT_TOL = 2e-3
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    pa.lib()


def _plan(b, target, override=None):
    return pa.pa_v2_plan(b.indptr, b.last_page_len, b.first_page_offset, b.page_size, b.num_qo_heads,
                         b.num_kv_heads, b.head_dim, pa.KV_DTYPES[b.dtype], target,
                         b.ppc_override if override is None else override, b.seq_lens)


def _close(a, b, tol):
    fin = torch.isfinite(b)
    assert torch.equal(torch.isfinite(a), fin)
    return float((a[fin] - b[fin]).abs().max()) <= tol if fin.any() else True


def _close_oracle(got, ref, tol):
    got = got.double().cpu().numpy()
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin)
    return float(np.abs(got[fin] - ref[fin]).max()) <= tol if fin.any() else True


@pytest.mark.parametrize("case", ["tiny_csr", "llama_8k", "sliding_window_batch", "one_chunk_per_request"])
def test_noalloc_matches_oracle_and_decode_twice(case):
    override = None
    if case == "tiny_csr":
        b, target = W.tiny_csr(), 1
    elif case == "llama_8k":
        b, target = W.llama3_8b_32k(context=8192), 152
    elif case == "sliding_window_batch":
        b, target = W.sliding_window_batch(), 304
    else:
        b, target = W.sliding_window_batch(), 1
        override = max(int(b.indptr[r + 1] - b.indptr[r]) for r in range(b.batch))
    plan = _plan(b, target, override)
    assert plan.needs_merge == (0 if case == "one_chunk_per_request" else 1)
    ref_o, ref_l = oracle.attention(b.q, b.k_pool, b.v_pool, b.indices, b.indptr, b.last_page_len,
                                    b.first_page_offset, b.scale)
    d = b.to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dec_o, dec_l = pa.pa_v2_decode(plan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len,
                                   d.first_page_offset, b.scale, status=status)
    dec_o, dec_l = dec_o.clone(), dec_l.clone()
    for _ in range(2):
        out = torch.full_like(dec_o, float("nan"))
        lse = torch.full_like(dec_l, float("nan"))
        pa.pa_v2_decode_noalloc(plan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len,
                                d.first_page_offset, b.scale, out=out, lse2_out=lse, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert _close_oracle(out, ref_o, OUT_TOL)
        assert _close_oracle(lse, ref_l, LSE_TOL)
        assert _close(out, dec_o, OUT_TOL)
        assert _close(lse, dec_l, LSE_TOL)


def test_noalloc_stacked_level_rows_land_out_row_step_apart():
    # cascade level 0: the members' heads stacked over the shared prefix (one request, stack_members = M),
    # member m written to row 2m of a [2M, Hq, D] buffer; rows 2m + 1 must stay untouched
    cb = W.cascade_shared_prefix(members=3, prefix_tokens=2048, suffix_range=(16, 64))
    b = cb.flat
    M, Hq, D = b.q.shape
    npre = len(cb.prefix_indices)
    dt = pa.KV_DTYPES[b.dtype]
    plan = pa.pa_v2_plan([0, npre], [b.page_size], [0], b.page_size, M * Hq, b.num_kv_heads, D, dt, 152, 0)
    plan.struct.stack_members = M
    plan.struct.out_row_step = 2
    assert plan.needs_merge == 1
    # the oracle: each member attends over the prefix pages alone
    ip = torch.arange(0, (M + 1) * npre, npre, dtype=torch.int32)
    idx = cb.prefix_indices.repeat(M)
    ref_o, ref_l = oracle.attention(b.q, b.k_pool, b.v_pool, idx, ip, torch.full((M,), b.page_size, dtype=torch.int32),
                                    torch.zeros(M, dtype=torch.int32), b.scale)
    d = b.to("cuda")
    pre = cb.prefix_indices.to("cuda")
    ip0 = torch.tensor([0, npre], dtype=torch.int32, device="cuda")
    lp0 = torch.tensor([b.page_size], dtype=torch.int32, device="cuda")
    fp0 = torch.zeros(1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        full_o = torch.full((2 * M, Hq, D), 7.0, device="cuda")
        full_l = torch.full((2 * M, Hq), 7.0, device="cuda")
        o, l = pa.pa_v2_decode_noalloc(plan, d.q, d.k_pool, d.v_pool, pre, ip0, lp0, fp0, b.scale,
                                       out=full_o[0::2], lse2_out=full_l[0::2], status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert o.shape == (M, Hq, D) and l.shape == (M, Hq)
        assert _close_oracle(full_o[0::2], ref_o, OUT_TOL)
        assert _close_oracle(full_l[0::2], ref_l, LSE_TOL)
        assert bool((full_o[1::2] == 7.0).all()) and bool((full_l[1::2] == 7.0).all())


def test_noalloc_empty_batch_launches_nothing():
    plan = pa.pa_v2_plan(torch.zeros(1, dtype=torch.int32), torch.zeros(0, dtype=torch.int32),
                         torch.zeros(0, dtype=torch.int32), 16, 32, 8, 128, pa.PA_F16, 152, 0)
    assert plan.num_chunks == 0
    q = torch.zeros(1, 32, 128, device="cuda")
    pool = torch.zeros(1, 16, 8, 128, dtype=torch.float16, device="cuda")
    idx = torch.zeros(1, dtype=torch.int32, device="cuda")
    ip = torch.zeros(1, dtype=torch.int32, device="cuda")
    none = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((1, 32, 128), 3.0, device="cuda")
    lse = torch.full((1, 32), 3.0, device="cuda")
    pa.pa_v2_decode_noalloc(plan, q, pool, pool, idx, ip, none, none, 0.125, out=out, lse2_out=lse)
    torch.cuda.synchronize()
    assert bool((out == 3.0).all()) and bool((lse == 3.0).all())


def test_noalloc_refuses_plans_beyond_its_array():
    # 16 requests of 4096 one-token pages in chunks of four pages: 16384 chunks x 8 heads x
    # 65 floats of workspace (about 34 MB), far beyond the fixed array
    B, pages = 16, 4096
    indptr = torch.arange(0, (B + 1) * pages, pages, dtype=torch.int32)
    plan = pa.pa_v2_plan(indptr, torch.ones(B, dtype=torch.int32), torch.zeros(B, dtype=torch.int32), 1, 8, 8, 64,
                         pa.PA_F16, 10 ** 9, 4)
    need = plan.counter_bytes + plan.workspace_v_bytes + plan.workspace_lse_bytes
    assert need > pa.NOALLOC_SCRATCH_BYTES
    q = torch.zeros(B, 8, 64, device="cuda")
    pool = torch.zeros(B * pages, 1, 8, 64, dtype=torch.float16, device="cuda")
    idx = torch.arange(B * pages, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PaError) as e:
        pa.pa_v2_decode_noalloc(plan, q, pool, pool, idx, indptr.cuda(), torch.ones(B, dtype=torch.int32).cuda(),
                                torch.zeros(B, dtype=torch.int32).cuda(), 0.125)
    assert e.value.status == pa.PA_ECAPACITY
