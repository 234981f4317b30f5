"""GPU parity: the C-ABI CUDA path against the f64 oracle, element by element.

Covers the five workloads at full size (in the launch configuration bench.py
times: plan target from the device's SM count and occupancy), a sweep over head
dims, GQA ratios, dtypes and page sizes with ragged lengths, mid-page window
starts and empty requests, chunk-size invariance, the merge kernel alone, and
the cascade composition.
"""
import ctypes
import math
import random
import zlib

import numpy as np
import pytest
import torch

import oracle
from paged_attention_decode_gb300 import pa_v2 as pa
from paged_attention_decode_gb300 import workloads as W
from parity_helpers import LSE_TOL, OUT_TOL, assert_close, check_batch, make_plan, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    pa.lib()


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------

def test_tiny_csr_fixed_chunks():
    b = W.tiny_csr()
    plan, *_ = check_batch(b, target=1)
    assert plan.num_chunks == 4 and plan.needs_merge == 1
    assert plan.request_indices.tolist() == [0, 0, 1, 1] and plan.kv_tile_indices.tolist() == [0, 1, 0, 1]


@pytest.fixture(scope="module")
def llama():
    return W.llama3_8b_32k()


def test_llama3_8b_32k_bench_launch(llama):
    """The launches bench.py can time: the device-derived target with the plan's own chunk-size search,
    and every size the autotuner may pick in its place with the same CTA count (108-112 pages; 112 gives
    each of the kernel's 8 warps 14 stages), the one-wave fit among them."""
    tgt = pa.pa_v2_default_target_ctas(32, 8, 128, 16, pa.PA_F16)
    plan, *_ = check_batch(llama)
    assert plan.needs_merge == 1 and plan.total_ctas == tgt
    fit = pa.pa_v2_wave_fit_pages_per_chunk(llama.indptr, plan.q_groups * plan.num_kv_heads, tgt)
    assert fit == 108 and plan.pages_per_chunk == 113
    for ppc in range(fit, plan.pages_per_chunk):
        p2, *_ = check_batch(llama, override=ppc, check_partials=False, fused=False)
        assert p2.total_ctas == tgt


@pytest.mark.parametrize("target", [640, 152, 10 ** 6])
def test_llama3_8b_32k_other_targets(llama, target):
    check_batch(llama, target=target, check_partials=(target == 152))


def test_sliding_window_batch():
    check_batch(W.sliding_window_batch())


@pytest.mark.parametrize("name", ["sliding_window_batch", "sparse_token_exact"])
def test_balanced_chunk_size_is_exact(name):
    """The chunk size bench.py takes for the paged workloads when the plan's search fits one wave:
    pa_v2_balanced_pages_per_chunk of the search's (72 for the sliding-window batch, the search's own
    228 for the sparse decode's one-wave fit), partials and merged output against the oracle."""
    b = W.WORKLOADS[name]()
    search = make_plan(b)
    ppc = search.pages_per_chunk
    if search.total_ctas > search.target_ctas:
        ppc = pa.pa_v2_wave_fit_pages_per_chunk(b.indptr, search.q_groups * search.num_kv_heads,
                                                search.target_ctas)
    bal = pa.pa_v2_balanced_pages_per_chunk(b.indptr, b.page_size, ppc)
    plan, *_ = check_batch(b, override=bal, fused=False)
    assert plan.num_chunks == make_plan(b, override=ppc).num_chunks


def test_sparse_token_exact_full():
    b = W.sparse_token_exact()
    check_batch(b)


def test_cascade_flat_and_two_level():
    cb = W.cascade_shared_prefix()
    f = cb.flat
    _, flat_o, flat_l, _ = check_batch(f, check_partials=False)
    co, cl = cascade_gpu(cb)
    ref_o, ref_l = oracle.attention(f.q, f.k_pool, f.v_pool, f.indices, f.indptr, f.last_page_len,
                                    f.first_page_offset, f.scale)
    assert_close(co, cl, ref_o, ref_l, "cascade")
    # the two levels partition the flat launch's key range: equal up to f32 rounding
    assert float((co - flat_o).abs().max()) <= 2 * OUT_TOL


@pytest.mark.parametrize("wave", [0, 40, 1000])
def test_cascade_driver_one_launch(wave):
    """The library's cascade path (pa_v2_cascade_plan + pa_v2_cascade_decode: both levels in one launch of
    the partial kernel, stacked level 0 read in place, rows interleaved for one merge); the device's wave
    split between the levels, a small one (few, long chunks) and a large one (many short chunks)."""
    from paged_attention_decode_gb300 import cascade as C
    cb = W.cascade_shared_prefix()
    f = cb.flat
    dt = pa.KV_DTYPES[f.dtype]
    M, Hq, D = f.q.shape
    fp1 = torch.zeros(M, dtype=torch.int32)
    cp = C.cascade_plan(len(cb.prefix_indices), cb.suffix_indptr, cb.suffix_last_page_len, fp1, f.page_size, Hq,
                        f.num_kv_heads, D, dt, wave, cb.suffix_lens)
    if wave:
        assert cp.level0.total_ctas + cp.level1.total_ctas <= max(wave, 8 + 8 * M)
    dev = "cuda"
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    args = (f.q.to(dev), f.k_pool.to(dev), f.v_pool.to(dev), cb.prefix_indices.to(dev), cb.suffix_indices.to(dev),
            cb.suffix_indptr.to(dev), cb.suffix_last_page_len.to(dev), fp1.to(dev), f.scale)
    out, lse = C.cascade_decode(cp, *args, status=status)
    out2, lse2 = C.cascade_decode(cp, *args, status=status)   # twice: counters and buffers reused
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_o, ref_l = oracle.cascade_ref(f.q, f.k_pool, f.v_pool, cb.prefix_indices, cb.suffix_indices,
                                      cb.suffix_indptr, cb.suffix_last_page_len, f.scale)
    assert_close(out, lse, ref_o, ref_l, "cascade driver")
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


@pytest.mark.parametrize("ps,D,dt", [(5, 64, torch.bfloat16), (8, 128, torch.float16), (32, 64, torch.bfloat16),
                                     (1, 128, torch.float16)])
def test_cascade_staging_paths_and_head_dims(ps, D, dt):
    """The two-level launch on every staging path of the tensor-core kernel: cp.async for page sizes TMA
    cannot stage (5, 1), TMA boxes of whole 8-row pages and 16-row slices of 32-row pages; head_dim 64 and
    128; against the oracle's cascade (levels + merge) and flat attention."""
    from paged_attention_decode_gb300 import cascade as C
    cb = W.cascade_shared_prefix(members=3, prefix_tokens=ps * (320 // ps), suffix_range=(3, 150), head_dim=D,
                                 page_size=ps, dtype=dt, seed=70 + ps)
    f = cb.flat
    M, Hq, _ = f.q.shape
    fp1 = torch.zeros(M, dtype=torch.int32)
    cp = C.cascade_plan(len(cb.prefix_indices), cb.suffix_indptr, cb.suffix_last_page_len, fp1, ps, Hq,
                        f.num_kv_heads, D, pa.KV_DTYPES[dt], 152, cb.suffix_lens)
    dev = "cuda"
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = C.cascade_decode(cp, f.q.to(dev), f.k_pool.to(dev), f.v_pool.to(dev), cb.prefix_indices.to(dev),
                                cb.suffix_indices.to(dev), cb.suffix_indptr.to(dev), cb.suffix_last_page_len.to(dev),
                                fp1.to(dev), f.scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_o, ref_l = oracle.cascade_ref(f.q, f.k_pool, f.v_pool, cb.prefix_indices, cb.suffix_indices,
                                      cb.suffix_indptr, cb.suffix_last_page_len, f.scale)
    assert_close(out, lse, ref_o, ref_l, f"cascade ps={ps} D={D}")
    flat_o, flat_l = oracle.attention(f.q, f.k_pool, f.v_pool, f.indices, f.indptr, f.last_page_len,
                                      f.first_page_offset, f.scale)
    assert_close(out, lse, flat_o, flat_l, f"cascade vs flat ps={ps} D={D}")


@pytest.mark.parametrize("members,Hq,Hkv,dt", [(2, 16, 4, torch.float16), (4, 32, 8, torch.bfloat16),
                                               (2, 32, 2, torch.float16), (3, 32, 2, torch.bfloat16)])
def test_cascade_level_tile_widths(members, Hq, Hkv, dt):
    """Each level of the one-launch cascade runs with its own n-tile count: 8 stacked heads at level 0 and
    4 at level 1 (one tile each), 16 and 4 (two and one), 32 and 16 (two tiles each, level 0 in two
    q-groups), 48 and 16; against the oracle's cascade and flat attention."""
    from paged_attention_decode_gb300 import cascade as C
    cb = W.cascade_shared_prefix(members=members, prefix_tokens=16 * 40, suffix_range=(20, 300), num_qo_heads=Hq,
                                 num_kv_heads=Hkv, head_dim=128, dtype=dt, seed=80 + members + Hkv)
    f = cb.flat
    M = f.q.shape[0]
    fp1 = torch.zeros(M, dtype=torch.int32)
    cp = C.cascade_plan(len(cb.prefix_indices), cb.suffix_indptr, cb.suffix_last_page_len, fp1, 16, Hq, Hkv, 128,
                        pa.KV_DTYPES[dt], 152, cb.suffix_lens)
    dev = "cuda"
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = C.cascade_decode(cp, f.q.to(dev), f.k_pool.to(dev), f.v_pool.to(dev), cb.prefix_indices.to(dev),
                                cb.suffix_indices.to(dev), cb.suffix_indptr.to(dev), cb.suffix_last_page_len.to(dev),
                                fp1.to(dev), f.scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_o, ref_l = oracle.cascade_ref(f.q, f.k_pool, f.v_pool, cb.prefix_indices, cb.suffix_indices,
                                      cb.suffix_indptr, cb.suffix_last_page_len, f.scale)
    assert_close(out, lse, ref_o, ref_l, f"cascade M={members} G={Hq // Hkv}")
    flat_o, flat_l = oracle.attention(f.q, f.k_pool, f.v_pool, f.indices, f.indptr, f.last_page_len,
                                      f.first_page_offset, f.scale)
    assert_close(out, lse, flat_o, flat_l, f"cascade vs flat M={members} G={Hq // Hkv}")


def test_cascade_row_map_past_the_merge_input_is_refused_on_the_device():
    """A part_rows entry pointing past the merge input: the kernel writes nothing there and records
    PA_DEVICE_BAD_INDPTR (the host cannot see device row maps)."""
    cb = W.cascade_shared_prefix(members=2, prefix_tokens=256, suffix_range=(20, 40))
    f = cb.flat
    M, Hq, D = f.q.shape
    dt = pa.KV_DTYPES[f.dtype]
    cps = pa.pa_v2_cascade_plan(M, len(cb.prefix_indices), cb.suffix_indptr, cb.suffix_last_page_len,
                                torch.zeros(M, dtype=torch.int32), f.page_size, Hq, f.num_kv_heads, D, dt, 152)
    dev = "cuda"
    pr0 = cps.l0_part_rows.clone()
    pr0[0] = cps.merge_rows + 1000
    merge_v = torch.zeros(cps.merge_rows, Hq, D, device=dev)
    merge_l = torch.zeros(cps.merge_rows, Hq, device=dev)
    canary = torch.full((4096,), 5.0, device=dev)   # allocated after the merge input
    lv0 = pa.cascade_level(cps.level0, cb.prefix_indices.to(dev), torch.tensor([0, len(cb.prefix_indices)],
                           dtype=torch.int32, device=dev), torch.tensor([f.page_size], dtype=torch.int32, device=dev),
                           torch.zeros(1, dtype=torch.int32, device=dev), pr0.to(dev))
    lv1 = pa.cascade_level(cps.level1, cb.suffix_indices.to(dev), cb.suffix_indptr.to(dev),
                           cb.suffix_last_page_len.to(dev), torch.zeros(M, dtype=torch.int32, device=dev),
                           cps.l1_part_rows.to(dev))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pa.pa_v2_cascade_decode(cps, lv0, lv1, f.q.to(dev), f.k_pool.to(dev), f.v_pool.to(dev), f.scale, merge_v, merge_l,
                            cps.merge_indptr.to(dev), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & pa.DEVICE_BAD_INDPTR
    assert bool((canary == 5.0).all())


@pytest.mark.parametrize("wave", [0, 24])
def test_cascade_on_a_mixed_batch(wave):
    """Detection + split + one two-level launch + merge on a batch with members, a mid-page sharer and
    strangers (row maps for both levels)."""
    from paged_attention_decode_gb300 import cascade as C
    b = W.cascade_mixed_batch()
    dt = pa.KV_DTYPES[b.dtype]
    cp = C.plan_batch(b.indptr, b.indices, b.last_page_len, b.first_page_offset, b.page_size, b.num_qo_heads,
                      b.num_kv_heads, b.head_dim, dt, wave_ctas=wave)
    assert cp is not None and cp.members == 3 and cp.shared_pages == b.meta["shared_pages"]
    d = b.to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = C.decode_batch(cp, d.q, d.k_pool, d.v_pool, b.scale, status=status)
    out2, lse2 = C.decode_batch(cp, d.q, d.k_pool, d.v_pool, b.scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref_o, ref_l = oracle.attention(b.q, b.k_pool, b.v_pool, b.indices, b.indptr, b.last_page_len,
                                    b.first_page_offset, b.scale)
    assert_close(out, lse, ref_o, ref_l, "mixed-batch cascade")
    assert torch.equal(out, out2)


@pytest.mark.parametrize("M,G", [(2, 4), (4, 4), (3, 2)])
def test_stacked_level0_reads_member_layout(M, G):
    """stack_members: one request over shared pages serves M members' heads, read and written in member
    layout; compared with the oracle on each member's own copy of the table."""
    Hkv, D, ps, npre = 2, 128, 16, 37
    g = torch.Generator().manual_seed(M * 10 + G)
    P = 2 * npre
    ids = torch.randperm(P, generator=g)[:npre].to(torch.int32)
    q = torch.randn(M, Hkv * G, D, generator=g)
    kp = torch.randn(P, ps, Hkv, D, generator=g).half()
    vp = torch.randn(P, ps, Hkv, D, generator=g).half()
    plan = pa.pa_v2_plan([0, npre], [ps], [0], ps, M * Hkv * G, Hkv, D, pa.PA_F16, 40)
    plan.struct.stack_members = M
    dev = "cuda"
    out, lse = pa.pa_v2_decode(plan, q.to(dev), kp.to(dev), vp.to(dev), ids.to(dev),
                               torch.tensor([0, npre], dtype=torch.int32, device=dev),
                               torch.tensor([ps], dtype=torch.int32, device=dev),
                               torch.zeros(1, dtype=torch.int32, device=dev), D ** -0.5)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.attention(q, kp, vp, ids.repeat(M), torch.arange(0, (M + 1) * npre, npre, dtype=torch.int32),
                                    [ps] * M, [0] * M, D ** -0.5)
    assert out.shape == (M, Hkv * G, D)
    assert_close(out, lse, ref_o, ref_l, "stacked level 0")


def cascade_gpu(cb):
    """Level 0 over the shared pages with stacked heads, level 1 over the suffixes, one merge."""
    f = cb.flat
    M, Hq, D = f.q.shape
    Hkv = f.num_kv_heads
    G = Hq // Hkv
    dev = "cuda"
    kp, vp = f.k_pool.to(dev), f.v_pool.to(dev)
    dt = pa.KV_DTYPES[f.dtype]
    npre = len(cb.prefix_indices)
    # level 0: one request, M*G query heads per KV head, h0 = kv*(M*G) + m*G + g
    q0 = f.q.to(dev).reshape(M, Hkv, G, D).permute(1, 0, 2, 3).reshape(1, Hkv * M * G, D).contiguous()
    ip0 = torch.tensor([0, npre], dtype=torch.int32)
    lp0 = torch.tensor([f.page_size], dtype=torch.int32)
    fp0 = torch.tensor([0], dtype=torch.int32)
    tgt0 = pa.pa_v2_default_target_ctas(M * Hq, Hkv, D, f.page_size, dt)
    p0 = pa.pa_v2_plan(ip0, lp0, fp0, f.page_size, M * Hq, Hkv, D, dt, tgt0)
    o0, l0 = pa.decode(p0, q0, kp, vp, cb.prefix_indices.to(dev), ip0.to(dev), lp0.to(dev), fp0.to(dev), f.scale)
    # level 1: each member's private suffix
    fp1 = torch.zeros(M, dtype=torch.int32)
    tgt1 = pa.pa_v2_default_target_ctas(Hq, Hkv, D, f.page_size, dt)
    p1 = pa.pa_v2_plan(cb.suffix_indptr, cb.suffix_last_page_len, fp1, f.page_size, Hq, Hkv, D, dt, tgt1)
    o1, l1 = pa.decode(p1, f.q.to(dev), kp, vp, cb.suffix_indices.to(dev), cb.suffix_indptr.to(dev),
                       cb.suffix_last_page_len.to(dev), fp1.to(dev), f.scale)
    # unstack level 0 and pair each member's two states
    o0 = o0.reshape(Hkv, M, G, D).permute(1, 0, 2, 3).reshape(M, Hq, D)
    l0 = l0.reshape(Hkv, M, G).permute(1, 0, 2).reshape(M, Hq)
    v_in = torch.stack([o0, o1], dim=1).reshape(2 * M, Hq, D).contiguous()
    lse_in = torch.stack([l0, l1], dim=1).reshape(2 * M, Hq).contiguous()
    oi = torch.arange(0, 2 * M + 1, 2, dtype=torch.int32, device=dev)
    out, lse = pa.pa_merge_states(v_in, lse_in, oi, M)
    torch.cuda.synchronize()
    return out, lse


# ---------------------------------------------------------------------------
# sweeps
# ---------------------------------------------------------------------------

SWEEP = [(dt, D, G, ps) for dt in (torch.float32, torch.float16, torch.bfloat16) for D in (64, 128)
         for G in (1, 2, 3, 4, 8, 16) for ps in (1, 4, 5, 8, 16, 32, 64)]


@pytest.mark.parametrize("dt,D,G,ps", SWEEP)
def test_sweep_ragged(dt, D, G, ps):
    rnd = random.Random(zlib.crc32(repr((str(dt), D, G, ps)).encode()))
    B = 4
    lens = [rnd.randint(1, 700), 0, rnd.randint(1, 40), rnd.randint(300, 1500)]
    fpos = [rnd.randrange(ps) if L else 0 for L in lens]
    Hkv = 2
    b = W.make_batch("sweep", lens, fpos, ps, num_qo_heads=Hkv * G, num_kv_heads=Hkv, head_dim=D, dtype=dt,
                     seed=rnd.randint(0, 10 ** 6), order="reversed" if G % 2 else "shuffled")
    check_batch(b, target=rnd.choice([1, 64, 700]), override=rnd.choice([0, 0, 1, 3]))


ONE_REQUEST = [(dt, D, ps) for dt in (torch.float16, torch.bfloat16) for D in (64, 128)
               for ps in (1, 4, 5, 8, 16, 32, 64, 256)]


@pytest.mark.parametrize("dt,D,ps", ONE_REQUEST)
def test_sweep_one_request(dt, D, ps):
    """One-request plans (the kernel's single-request geometry and its pre-wait L2 warm-up) on every
    staging path: cp.async for page sizes 1-5, TMA for 8, 16 and the multiples of 16; a window that
    starts mid-page and a ragged last page; several chunks."""
    rnd = random.Random(zlib.crc32(repr(("one", str(dt), D, ps)).encode()))
    G = rnd.choice([1, 2, 4, 8, 16])
    L = rnd.randint(40 * max(ps, 8), 60 * max(ps, 8))
    b = W.make_batch("one", [L], [rnd.randrange(ps)], ps, num_qo_heads=2 * G, num_kv_heads=2, head_dim=D,
                     dtype=dt, seed=rnd.randint(0, 10 ** 6), order="shuffled")
    plan, _, _, _ = check_batch(b, target=rnd.choice([64, 152, 700]), override=rnd.choice([0, 0, 3]))
    assert plan.batch == 1 and plan.num_chunks > 1


def test_plan_at_the_chunk_cap():
    """The largest plan the launch shape allows (PA_V2_MAX_CHUNKS = 65535 chunks, the pages' grid bound):
    21845 requests of three 8-row pages, windows starting and ending mid-page, one page per chunk; merged
    outputs, fused outputs and every chunk's partial against the oracle."""
    rnd = random.Random(65535)
    B = 21845
    fpos = [rnd.randrange(8) for _ in range(B)]
    lens = [rnd.randint(17 - f, 24 - f) for f in fpos]     # (fpo + len) in 17..24: exactly three pages
    b = W.make_batch("cap", lens, fpos, 8, 4, 1, 64, torch.float16, seed=7, slack=1.0)
    plan, _, _, _ = check_batch(b, target=1, override=1)
    assert plan.num_chunks == 65535 and plan.needs_merge


def test_chunk_size_invariance_seven_sizes():
    b = W.make_batch("inv", [4099, 77, 1, 2500], [5, 0, 0, 15], 16, 32, 8, 128, torch.float16, seed=5)
    outs = []
    for ppc in (1, 2, 3, 7, 16, 64, 1000):
        plan, o, lo, _ = check_batch(b, target=1, override=ppc, check_partials=(ppc in (1, 7)))
        outs.append(o)
    for o in outs[1:]:
        assert float((o - outs[0]).abs().max()) <= OUT_TOL


def test_empty_request_does_not_poison_neighbours():
    b = W.make_batch("empty", [300, 0, 0, 45], [0, 0, 0, 3], 16, 8, 2, 128, torch.bfloat16, seed=9)
    plan, o, lo, _ = check_batch(b, target=1000, override=1)
    assert torch.all(o[1:3] == 0) and torch.all(lo[1:3] == -math.inf)
    assert torch.isfinite(o).all() and torch.isfinite(lo[0]).all() and torch.isfinite(lo[3]).all()


def test_single_token_and_full_final_pages():
    # seq_len 1, a window that is exactly one full page, exactly full final pages
    b = W.make_batch("edge", [1, 16, 32, 17, 15], [0, 0, 0, 15, 1], 16, 4, 4, 64, torch.float16, seed=2)
    check_batch(b, target=1, override=1)
    check_batch(b, target=10 ** 6)


def test_nan_outside_sequences_is_never_read():
    """Pool entries outside every request are NaN: any stray read shows up in the output."""
    g = torch.Generator().manual_seed(4)
    lens, fpos = [70, 5, 33], [3, 0, 9]
    dk = [torch.randn(L, 2, 64, generator=g) for L in lens]
    dv = [torch.randn(L, 2, 64, generator=g) for L in lens]
    for dt in (torch.float16, torch.float32):
        for ps in (1, 4, 16, 32):
            fp = [f % ps for f in fpos]
            b = W.scatter_dense("nan", dk, dv, fp, ps, num_qo_heads=8, seed=ps, dtype=dt)
            check_batch(b, target=1, override=1)
            check_batch(b, target=10 ** 6)


@pytest.mark.parametrize("dt", [torch.float16, torch.bfloat16])
def test_cuda_core_kernel_on_16bit_pools(dt):
    """plan.kernel = 1 selects the CUDA-core kernel for 16-bit pools (groups of up to 8 heads)."""
    b = W.make_batch("simt16", [700, 33, 2100], [3, 0, 9], 16, 16, 2, 128, dt, seed=12)
    plan = make_plan(b, target=200)
    plan.struct.kernel = 1
    check_batch(b, plan=plan)


def test_plan_reuse_across_steps():
    """A plan stays valid while no request crosses a page boundary (PR #984, What changed 4)."""
    b = W.make_batch("reuse", [100, 200], [0, 0], 16, 8, 2, 128, torch.float16, seed=3)
    plan = make_plan(b, target=300)
    b2 = W.make_batch("reuse", [101, 201], [0, 0], 16, 8, 2, 128, torch.float16, seed=3)
    assert pa.pa_v2_plan_matches(plan, b2.indptr, b2.last_page_len, b2.first_page_offset)
    check_batch(b2, plan=plan)


# ---------------------------------------------------------------------------
# the merge kernel on its own
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("D", [64, 128, 6, 96, 256, 512, 200, 516])
def test_merge_states_alone(D):
    rng = np.random.default_rng(D)
    groups = [1, 3, 0, 5, 2, 1, 7]
    oi = np.concatenate([[0], np.cumsum(groups)]).astype(np.int32)
    N, H = int(oi[-1]), 3
    v = rng.standard_normal((N, H, D)).astype(np.float32)
    l = rng.uniform(-30, 30, (N, H)).astype(np.float32)
    l[4, 1] = -np.inf          # a -inf member contributes nothing
    v[4, 1] = 0
    l[9:11, :] = -np.inf       # an all-empty group (rows 9, 10 form group 4)
    v[9:11] = 0
    dev = "cuda"
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = pa.pa_merge_states(torch.from_numpy(v).to(dev), torch.from_numpy(l).to(dev),
                                  torch.from_numpy(oi).to(dev), len(groups), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref_o, ref_l = oracle.merge(v.astype(np.float64), l.astype(np.float64), oi)
    assert_close(out, lse, ref_o, ref_l, "merge")
    # a one-row group is an exact identity
    assert torch.equal(out[0].cpu(), torch.from_numpy(v[0]))
    assert torch.equal(lse[0].cpu(), torch.from_numpy(l[0]))


def test_merge_regrouping_is_associative_on_gpu():
    rng = np.random.default_rng(1)
    N, H, D = 12, 4, 128
    v = torch.from_numpy(rng.standard_normal((N, H, D)).astype(np.float32)).cuda()
    l = torch.from_numpy(rng.uniform(-10, 10, (N, H)).astype(np.float32)).cuda()
    full, fl = pa.pa_merge_states(v, l, torch.tensor([0, N], dtype=torch.int32, device="cuda"), 1)
    part, pl = pa.pa_merge_states(v, l, torch.tensor([0, 5, 6, N], dtype=torch.int32, device="cuda"), 3)
    again, al = pa.pa_merge_states(part, pl, torch.tensor([0, 3], dtype=torch.int32, device="cuda"), 1)
    torch.cuda.synchronize()
    assert float((again - full).abs().max()) <= 1e-5 and float((al - fl).abs().max()) <= 1e-5


# ---------------------------------------------------------------------------
# device-side bounds checks: bad device data is recorded in the status word, not read
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("ps", [16, 4])
def test_out_of_range_page_id_is_reported_not_read(ps):
    # page_size 16 stages with TMA (the box is redirected past the pool's end, which TMA
    # zero-fills); page_size 4 stages with cp.async (the copy is skipped)
    b = W.make_batch("badpage", [200, 90], [0, 3], ps, 8, 2, 128, torch.float16, seed=17)
    plan = make_plan(b, target=64)
    d = b.to("cuda")
    bad = d.indices.clone()
    bad[3] = b.num_pages
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_v2_decode(plan, d.q, d.k_pool, d.v_pool, bad, d.indptr, d.last_page_len, d.first_page_offset, b.scale,
                    status=status)
    torch.cuda.synchronize()
    word = int(status.item())
    assert word & pa.DEVICE_BAD_PAGE and pa.pa_status_from_device(word) == pa.PA_EOOB
    # every CTA still finished, so the ticket counters are back at zero and a clean call is exact
    assert int(plan.device_counters("cuda").abs().sum()) == 0
    check_batch(b, plan=plan, d=d)


def test_bad_o_indptr_is_reported():
    v = torch.randn(4, 2, 64, device="cuda")
    l = torch.randn(4, 2, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_merge_states(v, l, torch.tensor([0, 3, 2], dtype=torch.int32, device="cuda"), 2, status=status)
    pa.pa_merge_states(v, l, torch.tensor([0, 9], dtype=torch.int32, device="cuda"), 1, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & pa.DEVICE_BAD_INDPTR


def test_out_of_range_request_index_is_reported():
    # two requests: a one-request plan fixes every chunk's request and reads no chunk arrays
    b = W.make_batch("badreq", [300, 40], [0, 0], 16, 8, 2, 128, torch.float16, seed=18)
    plan = make_plan(b, target=16)
    d = b.to("cuda")
    ri, ti, _ = plan.device_arrays("cuda")
    bad_ri = ri.clone()
    bad_ri[0] = 7
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_v2_decode_partial(plan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len,
                            d.first_page_offset, b.scale, status=status, request_indices=bad_ri,
                            kv_tile_indices=ti)
    torch.cuda.synchronize()
    assert int(status.item()) & pa.DEVICE_BAD_REQUEST


# ---------------------------------------------------------------------------
# chunk-size autotuner: real timed launches, and the tuned plan is still exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fused", [False, True])
def test_autotune_times_candidates_and_tuned_plan_is_exact(fused):
    from paged_attention_decode_gb300 import autotune
    b = W.make_batch("tune", [3000, 700, 1, 0], [0, 5, 0, 0], 16, 8, 2, 128, torch.float16, seed=19)
    res = autotune.tune(b, "cuda", reps=3, fused=fused)
    assert res.default_pages_per_chunk in res.times_us
    assert res.pages_per_chunk in res.times_us
    assert all(t > 0 for t in res.times_us.values())
    check_batch(b, override=res.pages_per_chunk)


# ---------------------------------------------------------------------------
# one step from host buffers (pa_v2_decode_host)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("name", ["tiny_csr", "sliding_window_batch", "nomerge"])
@pytest.mark.parametrize("graph", [False, True])
@pytest.mark.parametrize("mapped", [False, True])
def test_host_step_matches_the_device_path(name, graph, mapped):
    if name == "nomerge":
        b = W.make_batch("nomerge", [40, 17, 0], [0, 3, 0], 16, 8, 2, 128, torch.float16, seed=23)
        plan = make_plan(b, target=1)
        assert not plan.needs_merge
    else:
        b = W.WORKLOADS[name]()
        plan = make_plan(b)
    d = b.to("cuda")
    step = pa.HostStep(plan, d.k_pool, d.v_pool, graph_scale=b.scale if graph else None, mapped=mapped)
    step.pack(b.q, b.indices, b.indptr, b.last_page_len, b.first_page_offset)
    for _ in range(2):                                  # the status slot is re-zeroed by every step
        o, l = step.run(b.scale)
    ref_o, ref_l = oracle.attention(b.q, b.k_pool, b.v_pool, b.indices, b.indptr, b.last_page_len,
                                    b.first_page_offset, b.scale)
    assert_close(o.clone(), l.clone(), ref_o, ref_l, f"host step {name}")
    o2, l2 = pa.decode(plan, d.q, d.k_pool, d.v_pool, d.indices, d.indptr, d.last_page_len, d.first_page_offset,
                       b.scale)
    assert torch.equal(o2.cpu(), o) and torch.equal(l2.cpu(), l)


@pytest.mark.parametrize("graph", [False, True])
@pytest.mark.parametrize("mapped", [False, True])
def test_host_step_refuses_a_stale_plan_and_reports_bad_pages(graph, mapped):
    b = W.make_batch("hs", [100, 60], [0, 0], 16, 8, 2, 128, torch.float16, seed=24)
    plan = make_plan(b, target=16)
    d = b.to("cuda")
    step = pa.HostStep(plan, d.k_pool, d.v_pool, graph_scale=b.scale if graph else None, mapped=mapped)
    grown = W.make_batch("hs", [100, 90], [0, 0], 16, 8, 2, 128, torch.float16, seed=24)
    step.pack(grown.q, grown.indices[:b.indices.numel()], grown.indptr, grown.last_page_len,
              grown.first_page_offset)
    with pytest.raises(pa.PaError) as e:
        step.run(b.scale)
    assert e.value.status == pa.PA_EGEOMETRY
    bad = b.indices.clone()
    bad[2] = b.num_pages
    step.pack(b.q, bad, b.indptr, b.last_page_len, b.first_page_offset)
    with pytest.raises(pa.PaError) as e:
        step.run(b.scale)
    assert e.value.status == pa.PA_EOOB
    step.pack(b.q, b.indices, b.indptr, b.last_page_len, b.first_page_offset)
    o, l = step.run(b.scale)                            # a clean step afterwards is exact again
    ref_o, ref_l = oracle.attention(b.q, b.k_pool, b.v_pool, b.indices, b.indptr, b.last_page_len,
                                    b.first_page_offset, b.scale)
    assert_close(o.clone(), l.clone(), ref_o, ref_l, "host step after errors")


@pytest.mark.parametrize("mapped", [False, True])
def test_host_graph_replays_new_inputs_and_other_scales_take_the_direct_path(mapped):
    """The graph binds buffers and scale; each run reads the step's current host inputs (mapped: the kernels
    read them from host memory, written by the host between steps)."""
    sets = [W.make_batch("hg", [300, 200], [0, 5], 16, 8, 2, 128, torch.float16, seed=s) for s in (31, 32)]
    b0 = sets[0]
    plan = make_plan(b0, target=32)
    d = b0.to("cuda")
    step = pa.HostStep(plan, d.k_pool, d.v_pool, graph_scale=b0.scale, mapped=mapped)
    for b in sets:  # same geometry and pool; new q and a new page permutation of the same pool
        q = b.q
        step.pack(q, b0.indices.flip(0).contiguous(), b0.indptr, b0.last_page_len, b0.first_page_offset)
        for scale in (b0.scale, 0.5 * b0.scale):
            o, l = step.run(scale)
            ref_o, ref_l = oracle.attention(q, b0.k_pool, b0.v_pool, b0.indices.flip(0).contiguous(), b0.indptr,
                                            b0.last_page_len, b0.first_page_offset, scale)
            assert_close(o.clone(), l.clone(), ref_o, ref_l, f"host graph scale {scale}")


@pytest.mark.parametrize("graph", [False, True])
def test_mapped_host_steps_return_complete_results(graph):
    """The copy-free calls return once the merge's CTA count in the status slot is complete, before the
    launch has formally finished: read straight after each of 40 consecutive steps (two input sets in turn,
    so a step that returned early would still show the other set's results), every output must equal the
    device path's for that step's inputs, bit for bit."""
    sets = [W.make_batch("hc", [700, 300, 45], [3, 0, 9], 16, 8, 2, 128, torch.float16, seed=s) for s in (41, 42)]
    b0 = sets[0]
    plan = make_plan(b0, target=64)
    assert plan.needs_merge
    d = b0.to("cuda")
    step = pa.HostStep(plan, d.k_pool, d.v_pool, graph_scale=b0.scale if graph else None, mapped=True)
    tables = [b0.indices, b0.indices.flip(0).contiguous()]
    want = []
    for b, tab in zip(sets, tables):
        o, l = pa.decode(plan, b.q.cuda(), d.k_pool, d.v_pool, tab.cuda(), d.indptr, d.last_page_len,
                         d.first_page_offset, b0.scale)
        want.append((o.cpu(), l.cpu()))
    for i in range(40):
        b, tab = sets[i % 2], tables[i % 2]
        step.pack(b.q, tab, b0.indptr, b0.last_page_len, b0.first_page_offset)
        o, l = step.run(b0.scale)
        assert torch.equal(o, want[i % 2][0]) and torch.equal(l, want[i % 2][1]), f"step {i}"
    torch.cuda.synchronize()


def test_mapped_host_step_refuses_unaligned_buffers():
    """The copy-free calls need 16-byte aligned host buffers; an unaligned one is refused before any launch."""
    b = W.make_batch("hm", [40, 17], [0, 3], 16, 8, 2, 128, torch.float16, seed=25)
    plan = make_plan(b, target=8)
    d = b.to("cuda")
    step = pa.HostStep(plan, d.k_pool, d.v_pool, mapped=True)
    step.pack(b.q, b.indices, b.indptr, b.last_page_len, b.first_page_offset)
    ri, ti, oi = plan.device_arrays(d.q.device)
    ws_v, ws_l = step.ws
    big = torch.zeros(step.in_bytes + 16, dtype=torch.uint8).pin_memory()
    big[4:4 + step.in_bytes] = step.host_in          # the same words, 4 bytes off a 16-byte boundary
    L = pa.lib()
    args = (d.k_pool.data_ptr(), d.v_pool.data_ptr(), pa.KV_DTYPES[d.k_pool.dtype], d.k_pool.shape[0],
            ri.data_ptr(), ti.data_ptr(), oi.data_ptr(), float(b.scale), ws_v.data_ptr(), ws_l.data_ptr())
    stream = torch.cuda.current_stream().cuda_stream
    assert L.pa_v2_decode_host_mapped(ctypes.byref(plan.struct), big.data_ptr() + 4, step.host_out.data_ptr(),
                                      *args, stream) == pa.PA_EINVAL
    g = ctypes.c_void_p()
    assert L.pa_v2_host_graph_create_mapped(ctypes.byref(plan.struct), step.host_in.data_ptr(),
                                            step.host_out.data_ptr() + 4, *args, ctypes.byref(g)) == pa.PA_EINVAL
    assert not g.value
    o, l = step.run(b.scale)                          # the aligned buffers still work
    ref_o, ref_l = oracle.attention(b.q, b.k_pool, b.v_pool, b.indices, b.indptr, b.last_page_len,
                                    b.first_page_offset, b.scale)
    assert_close(o.clone(), l.clone(), ref_o, ref_l, "mapped host step")
