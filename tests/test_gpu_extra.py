"""GPU: the second-K-stream partial kernels (pa_v2_decode_partial_extra) against the oracle -- partials
chunk by chunk and the merged result -- on MLA-shaped (values = latent rows) and separate-V inputs,
token-exact and paged tables, f16 and bf16, and the DSA-shaped workload.  plan.kernel 0 runs the
tensor-memory kernel (values in the key tile; separate values fall back to the warp-level tensor-core
kernel), 1 the CUDA-core kernel, 2 the warp-level tensor-core kernel."""
import math

import pytest
import torch

import oracle
from paged_attention_decode_gb300 import pa_v2 as pa
from paged_attention_decode_gb300 import workloads as W
from parity_helpers import assert_close

pytestmark = pytest.mark.gpu

D, E = 512, 64


def _paged(seq, fpo, ps, Hq, Hkv, dtype, seed, k_width=640, v_width=None, shared_v=True):
    """A paged batch whose k rows are k_width wide (key = first 512), extra rows 64 wide."""
    b = W.make_batch("extra", seq, fpo, ps, Hq, Hkv, k_width, dtype, seed=seed)
    gen = torch.Generator().manual_seed(seed + 7)
    b.q = torch.randn(len(seq), Hq, D, generator=gen)
    qe = torch.randn(len(seq), Hq, E, generator=gen)
    ke = torch.randn(b.k_pool.shape[0], ps, Hkv, E, generator=gen).to(dtype)
    if shared_v:
        b.v_pool = b.k_pool
    elif v_width is not None:
        b.v_pool = torch.randn(b.k_pool.shape[0], ps, Hkv, v_width, generator=gen).to(dtype)
    b.head_dim = D
    return W.ExtraStreamBatch(b, qe, ke, D, shared_v)


def _check(x, target=None, override=0, scale=None, kernel=0):
    b = x.batch
    dt = pa.KV_DTYPES[b.dtype]
    tgt = target or pa.pa_v2_default_target_ctas(b.num_qo_heads, b.num_kv_heads, D, b.page_size, dt)
    plan = pa.pa_v2_plan(b.indptr, b.last_page_len, b.first_page_offset, b.page_size, b.num_qo_heads,
                         b.num_kv_heads, D, dt, tgt, override, b.seq_lens)
    plan.struct.kernel = kernel
    scale = scale or 1.0 / math.sqrt(D + E)
    d = x.to("cuda")
    db = d.batch
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    v, l = pa.pa_v2_decode_partial_extra(plan, db.q, d.q_extra, db.k_pool, db.v_pool, d.k_extra_pool, db.indices,
                                         db.indptr, db.last_page_len, db.first_page_offset, scale, status=status)
    out, lse = pa.decode_extra(plan, db.q, d.q_extra, db.k_pool, db.v_pool, d.k_extra_pool, db.indices, db.indptr,
                               db.last_page_len, db.first_page_offset, scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    pv, pl = oracle.partials_extra(b.q, x.q_extra, b.k_pool, x.k_extra_pool, b.v_pool, D, b.indices, b.indptr,
                                   b.last_page_len, b.first_page_offset, scale, plan.pages_per_chunk,
                                   plan.request_indices, plan.kv_tile_indices)
    assert_close(v[:plan.num_chunks], l[:plan.num_chunks], pv, pl, f"partials ppc={plan.pages_per_chunk}")
    ro, rl = oracle.attention_extra(b.q, x.q_extra, b.k_pool, x.k_extra_pool, b.v_pool, D, b.indices, b.indptr,
                                    b.last_page_len, b.first_page_offset, scale)
    assert_close(out, lse, ro, rl, "merged")
    return plan


@pytest.mark.parametrize("kernel", [0, 1, 2])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("ps,seq,fpo,override", [(1, [300, 77, 0, 1], [0, 0, 0, 0], 64),
                                                 (16, [500, 33, 16], [3, 0, 15], 4),
                                                 (64, [700, 64, 1], [10, 0, 0], 3),
                                                 (5, [123, 40], [4, 2], 7)])
def test_mla_shape_parity(dtype, ps, seq, fpo, override, kernel):
    _check(_paged(seq, fpo, ps, 32, 1, dtype, seed=31 + ps), override=override, kernel=kernel)


@pytest.mark.parametrize("kernel", [0, 2])
@pytest.mark.parametrize("G", [4, 16, 20, 40])
def test_group_sizes_and_kv_heads(G, kernel):
    """Partial last q-groups (G = 20: 8 + 8 + 4 heads for the 8-head kernels; G = 40: 32 + 8 for the
    tensor-memory kernel) and two KV heads."""
    _check(_paged([200, 95], [0, 1], 16, 2 * G, 2, torch.bfloat16, seed=40 + G), override=5, kernel=kernel)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("ps,seq,fpo,override", [(1, [3000, 129, 128, 127], [0, 0, 0, 0], 1000),
                                                 (256, [900, 300], [200, 0], 2),
                                                 (16, [2100], [7], 80)])
def test_multi_tile_chunks(dtype, ps, seq, fpo, override):
    """Chunks of several 128-row tiles (the tensor-memory kernel's refill pipeline), tile-sized and
    one-off-tile-sized requests, and a 256-row page whose first tile is all before first_page_offset."""
    _check(_paged(seq, fpo, ps, 32, 1, dtype, seed=80 + ps), override=override)


@pytest.mark.parametrize("kernel", [0, 2])
def test_rising_scores_rescale_the_accumulator(kernel):
    """Extra-key rows grow with their position (the values do not), so the tiles' maximum scores climb
    by several times 8 (log2 units) along the chunk: the tensor-memory kernel raises its running
    maxima and rescales O^T and the row sums in place, repeatedly."""
    x = _paged([1400], [0], 1, 32, 1, torch.bfloat16, seed=90)
    ke = x.k_extra_pool.float()
    rows = x.batch.indices[:1400].long()         # page_size 1: token t is pool row indices[t]
    ke[rows] *= (1.0 + torch.arange(1400, dtype=torch.float32) / 32.0).view(-1, 1, 1, 1)
    x.k_extra_pool = ke.to(torch.bfloat16)
    _check(x, override=1400, kernel=kernel)


@pytest.mark.parametrize("kernel", [0, 1, 2])
def test_separate_values_and_row_strides(kernel):
    x = _paged([180, 40], [2, 0], 16, 16, 1, torch.float16, seed=50, k_width=520, v_width=528, shared_v=False)
    _check(x, override=4, kernel=kernel)


def test_plan_default_target_and_empty_requests():
    _check(_paged([0, 1500, 0, 9], [0, 0, 0, 5], 16, 64, 1, torch.bfloat16, seed=60))


@pytest.mark.parametrize("kernel", [0, 1, 2])
def test_dsa_shaped_workload(kernel):
    x = W.dsa_sparse_decode(batch=2, kv_len=4096, topk=2048)
    _check(x, scale=x.batch.scale, kernel=kernel)


def test_head_dim_512_plans_are_refused_by_the_single_stream_kernel():
    x = _paged([64], [0], 16, 16, 1, torch.float16, seed=70)
    b = x.batch
    plan = pa.pa_v2_plan(b.indptr, b.last_page_len, b.first_page_offset, 16, 16, 1, D, pa.PA_F16, 8, 0, b.seq_lens)
    d = x.to("cuda").batch
    with pytest.raises(pa.PaError) as e:
        pa.pa_v2_decode_partial(plan, d.q, d.k_pool[..., :D].contiguous(), d.k_pool[..., :D].contiguous(), d.indices,
                                d.indptr, d.last_page_len, d.first_page_offset, 0.1)
    assert e.value.status == pa.PA_EUNSUPPORTED


def test_out_of_range_page_id_is_reported_by_the_second_k_stream_kernels():
    for kernel in (0, 2):
        x = _paged([300, 90], [0, 0], 1, 32, 1, torch.bfloat16, seed=95)
        b = x.batch
        dt = pa.KV_DTYPES[b.dtype]
        plan = pa.pa_v2_plan(b.indptr, b.last_page_len, b.first_page_offset, 1, 32, 1, D, dt, 16, 0, b.seq_lens)
        plan.struct.kernel = kernel
        d = x.to("cuda")
        db = d.batch
        bad = db.indices.clone()
        bad[5] = b.k_pool.shape[0]          # one past the pool
        bad[310] = -3
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        pa.pa_v2_decode_partial_extra(plan, db.q, d.q_extra, db.k_pool, db.v_pool, d.k_extra_pool, bad, db.indptr,
                                      db.last_page_len, db.first_page_offset, 0.05, status=status)
        torch.cuda.synchronize()
        word = int(status.item())
        assert word & pa.DEVICE_BAD_PAGE and pa.pa_status_from_device(word) == pa.PA_EOOB, (kernel, word)
    # the context is still usable and a clean call is exact
    _check(_paged([300, 90], [0, 0], 1, 32, 1, torch.bfloat16, seed=95), override=64)


def test_bounded_wait_gives_up_and_the_other_role_follows():
    """The tensor-memory kernel's wait: one warp's wait times out after ~2^20 cycles and raises the abort
    flag; the other warp, waiting with the full ~2^31-cycle limit, leaves through the flag long before it."""
    import time
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    completed = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    pa.pa_v2_selftest_wait(status, completed, 1 << 20)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(status.item()) == pa.DEVICE_WAIT_TIMEOUT
    assert pa.pa_status_from_device(int(status.item())) == pa.PA_ECUDA
    assert completed.tolist() == [0, 0]
    assert elapsed < 0.5, elapsed
    with pytest.raises(pa.PaError):
        pa.pa_v2_selftest_wait(status, completed, 10)
    _check(_paged([200], [0], 1, 32, 1, torch.bfloat16, seed=96), override=128)
