"""pa_v2_decode_noalloc against pa_v2_decode (GPU).

Some callers cannot allocate device memory -- for example a serving engine that
has reserved the whole GPU for its own pools, or a plugin that its host hands
only input and output pointers -- so they cannot supply the workspace and
ticket counters pa_v2_decode needs.  pa_v2_decode_noalloc takes both from the
library's fixed device array instead.  These tests call it through the C ABI,
twice in a row on the same array, and compare each result with pa_v2_decode on
the same inputs; they also check that a plan too large for the array is
refused before any launch.  The file sorts last so that a run stopping at the
first failure has already run every other test.
"""
import pytest
import torch

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


def _plan(b, target):
    return pa.pa_v2_plan(b.indptr, b.last_page_len, b.first_page_offset, b.page_size, b.num_qo_heads,
                         b.num_kv_heads, b.head_dim, pa.KV_DTYPES[b.dtype], target, b.ppc_override, b.seq_lens)


def _close(a, b, tol):
    fin = torch.isfinite(b)
    assert torch.equal(torch.isfinite(a), fin)
    return float((a[fin] - b[fin]).abs().max()) <= tol if fin.any() else True


@pytest.mark.parametrize("case", ["tiny_csr", "llama_8k", "sliding_window_batch"])
def test_noalloc_matches_decode_twice(case):
    if case == "tiny_csr":
        b, target = W.tiny_csr(), 1
    elif case == "llama_8k":
        b, target = W.llama3_8b_32k(context=8192), 152
    else:
        b, target = W.sliding_window_batch(), 304
    plan = _plan(b, target)
    assert plan.needs_merge == 1
    d = b.to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref_o, ref_l = pa.pa_v2_decode(plan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len,
                                   d.first_page_offset, b.scale, status=status)
    ref_o, ref_l = ref_o.clone(), ref_l.clone()
    for _ in range(2):
        out = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_l, float("nan"))
        pa.pa_v2_decode_noalloc(plan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len,
                                d.first_page_offset, b.scale, out=out, lse2_out=lse, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert _close(out, ref_o, OUT_TOL)
        assert _close(lse, ref_l, LSE_TOL)


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
