"""Host-side checks of the C ABI (no GPU needed).

- libpa_v2.so loads and exports every function include/pa_v2.h declares;
- pa_v2_plan (binary search) is bit-exact against the oracle plan (linear scan)
  on the worked examples and on random geometries;
- every host-side rejection path returns its status before any launch;
- the plan's reuse predicate and the q-heads-per-CTA rule.
"""
import os
import random
import re

import numpy as np
import pytest
import torch

import oracle
from paged_attention_decode_gb300 import build as pa_build
from paged_attention_decode_gb300 import pa_v2 as pa
from paged_attention_decode_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    pa_build.build()


def _header_functions():
    text = open(os.path.join(ROOT, "include", "pa_v2.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(pa_[a-z0-9_]+)\s*\(", text,
                                 flags=re.M)))


def test_library_exports_every_declared_function():
    declared = _header_functions()
    assert len(declared) >= 9, declared
    L = pa.lib()
    for name in declared:
        assert hasattr(L, name), name
    assert sorted(pa.ABI_SYMBOLS) == declared
    assert "sm_103a" in pa.pa_version()


def test_status_strings_and_device_status_mapping():
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert pa.pa_status_string(code).startswith("PA_")
    assert pa.pa_status_from_device(0) == pa.PA_OK
    assert pa.pa_status_from_device(pa.DEVICE_BAD_PAGE) == pa.PA_EOOB
    assert pa.pa_status_from_device(pa.DEVICE_BAD_INDPTR | pa.DEVICE_BAD_SLOT) == pa.PA_EOOB
    assert pa.pa_status_from_device(pa.DEVICE_WAIT_TIMEOUT) == pa.PA_ECUDA


def expected_hpc(G, dtype=pa.PA_F16):
    """Documented rule: a CTA serves up to 16 query heads of one KV head with f16/bf16 pools
    (tensor-core kernel) and up to 8 with f32 pools (CUDA-core kernel)."""
    return min(G, 8 if dtype == pa.PA_F32 else 16)


@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 8, 12, 16, 32])
def test_q_heads_per_cta_rule(G):
    for D in (64, 128):
        for dt in (pa.PA_F32, pa.PA_F16, pa.PA_BF16):
            assert pa.pa_v2_q_heads_per_cta(G, D, dt) == expected_hpc(G, dt)
    assert pa.pa_v2_q_heads_per_cta(G, 96, pa.PA_F16) == 0
    assert pa.pa_v2_q_heads_per_cta(G, 128, 7) == 0
    assert pa.pa_v2_q_heads_per_cta(0, 128, pa.PA_F16) == 0


def _oracle_plan(indptr, Hq, Hkv, target, override=0, dtype=pa.PA_F16):
    G = Hq // Hkv
    qg = -(-G // expected_hpc(G, dtype))
    return oracle.plan(indptr, Hkv, qg, target, override)


def _assert_same_plan(p, ref, batch):
    assert p.pages_per_chunk == ref.pages_per_chunk
    assert p.lo_pages_per_chunk == ref.lo and p.hi_pages_per_chunk == ref.hi
    assert p.num_chunks == ref.num_chunks
    assert np.array_equal(p.request_indices.numpy(), ref.request_indices)
    assert np.array_equal(p.kv_tile_indices.numpy(), ref.kv_tile_indices)
    assert np.array_equal(p.o_indptr.numpy(), ref.o_indptr)
    assert p.needs_merge == int(ref.num_chunks > batch)


def test_plan_matches_oracle_on_workloads():
    cases = [(W.tiny_csr(), 1, 2), (W.sliding_window_batch(), 640, 0),
             (W.sparse_token_exact(cap=8192, selected=2048, heads=8), 456, 0)]
    for b, target, override in cases:
        override = override or b.ppc_override
        p = pa.pa_v2_plan(b.indptr, b.last_page_len, b.first_page_offset, b.page_size, b.num_qo_heads,
                          b.num_kv_heads, b.head_dim, pa.KV_DTYPES[b.dtype], target, override, b.seq_lens)
        ref = _oracle_plan(b.indptr, b.num_qo_heads, b.num_kv_heads, target, override, pa.KV_DTYPES[b.dtype])
        _assert_same_plan(p, ref, b.batch)
        assert p.workspace_v_bytes == p.num_chunks * b.num_qo_heads * b.head_dim * 4
        assert p.workspace_lse_bytes == p.num_chunks * b.num_qo_heads * 4
        assert p.total_ctas == p.num_chunks * b.num_kv_heads * p.q_groups


def test_plan_tiny_worked_example():
    b = W.tiny_csr()
    p = pa.pa_v2_plan(b.indptr, b.last_page_len, b.first_page_offset, 4, 4, 2, 64, pa.PA_F32, 1, 2)
    assert p.num_chunks == 4 and p.needs_merge == 1
    assert p.request_indices.tolist() == [0, 0, 1, 1]
    assert p.kv_tile_indices.tolist() == [0, 1, 0, 1]
    assert p.o_indptr.tolist() == [0, 2, 4]


def test_plan_llama_context_targets():
    indptr = [0, 2048]
    for target, ppc, n in ((640, 25, 82), (304, 55, 38)):
        p = pa.pa_v2_plan(indptr, [16], [0], 16, 32, 8, 128, pa.PA_F16, target)
        assert (p.pages_per_chunk, p.num_chunks) == (ppc, n)


def test_plan_binary_search_equals_linear_scan_random():
    rng = random.Random(7)
    for case in range(400):
        B = rng.randint(1, 10)
        ps = rng.choice([1, 4, 16, 32])
        lens = [rng.choice([0, 1, rng.randint(1, 5000), rng.randint(1, 200000) if ps == 16 else 7]) for _ in range(B)]
        fpos = [rng.randrange(ps) if L else 0 for L in lens]
        geo = [W.page_geometry(L, f, ps) for L, f in zip(lens, fpos)]
        indptr = np.concatenate([[0], np.cumsum([g[0] for g in geo])]).astype(np.int32)
        lpl = [g[1] for g in geo]
        Hkv = rng.choice([1, 2, 8])
        Hq = Hkv * rng.choice([1, 2, 4, 8, 12, 16])
        target = rng.randint(1, 3000)
        override = rng.choice([0, 0, 0, 1, rng.randint(1, 300)])
        try:
            ref = _oracle_plan(indptr, Hq, Hkv, target, override)
        except ValueError:
            with pytest.raises(pa.PaError):
                pa.pa_v2_plan(indptr, lpl, fpos, ps, Hq, Hkv, 128, pa.PA_F16, target, override, lens)
            continue
        p = pa.pa_v2_plan(indptr, lpl, fpos, ps, Hq, Hkv, 128, pa.PA_F16, target, override, lens)
        _assert_same_plan(p, ref, B)


def test_plan_grid_floor():
    pages = [40] * 4000
    indptr = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
    p = pa.pa_v2_plan(indptr, [16] * 4000, [0] * 4000, 16, 8, 8, 128, pa.PA_F16, 10 ** 9)
    assert p.lo_pages_per_chunk == 3 and p.pages_per_chunk == 3 and p.num_chunks == 56000
    with pytest.raises(pa.PaError) as e:
        pa.pa_v2_plan(indptr, [16] * 4000, [0] * 4000, 16, 8, 8, 128, pa.PA_F16, 1, 1)   # override too small
    assert e.value.status == pa.PA_EINVAL
    many = np.arange(0, 70001, dtype=np.int32)      # 70000 one-page requests cannot fit 65535 chunks
    with pytest.raises(pa.PaError) as e:
        pa.pa_v2_plan(many, [1] * 70000, [0] * 70000, 16, 8, 8, 128, pa.PA_F16, 1)
    assert e.value.status == pa.PA_EINVAL


def test_plan_empty_and_degenerate_batches():
    p = pa.pa_v2_plan([0, 0, 3, 3], [0, 3, 0], [0, 2, 0], 4, 4, 4, 64, pa.PA_F16, 10 ** 6)
    assert p.request_indices.tolist() == [0, 1, 1, 1, 2] and p.o_indptr.tolist() == [0, 1, 4, 5]
    p0 = pa.pa_v2_plan([0], [], [], 16, 8, 8, 128, pa.PA_F16, 100)
    assert p0.num_chunks == 0 and p0.needs_merge == 0


@pytest.mark.parametrize("mut,code", [
    (dict(indptr=[1, 4, 7]), pa.PA_EGEOMETRY),
    (dict(indptr=[0, 4, 3]), pa.PA_EGEOMETRY),
    (dict(lpl=[0, 1]), pa.PA_EGEOMETRY),
    (dict(lpl=[5, 1]), pa.PA_EGEOMETRY),
    (dict(fpo=[4, 2]), pa.PA_EGEOMETRY),
    (dict(seq_lens=[13, 8]), pa.PA_EGEOMETRY),
    (dict(head_dim=96), pa.PA_EUNSUPPORTED),
    (dict(kv_dtype=9), pa.PA_EUNSUPPORTED),
    (dict(page_size=24), pa.PA_EUNSUPPORTED),
    (dict(heads=(6, 4)), pa.PA_EINVAL),
    (dict(target=0), pa.PA_EINVAL),
])
def test_plan_rejections(mut, code):
    args = dict(indptr=[0, 4, 7], lpl=[1, 1], fpo=[0, 2], seq_lens=[13, 7], head_dim=64, kv_dtype=pa.PA_F32,
                page_size=4, heads=(4, 2), target=8)
    args.update(mut)
    with pytest.raises(pa.PaError) as e:
        pa.pa_v2_plan(args["indptr"], args["lpl"], args["fpo"], args["page_size"], args["heads"][0],
                      args["heads"][1], args["head_dim"], args["kv_dtype"], args["target"], 0, args["seq_lens"])
    assert e.value.status == code


def test_plan_capacity_error_reports_need():
    import ctypes
    st = pa.PlanStruct()
    ip = torch.tensor([0, 10], dtype=torch.int32)
    lp = torch.tensor([16], dtype=torch.int32)
    fp = torch.tensor([0], dtype=torch.int32)
    ri = torch.zeros(2, dtype=torch.int32)
    oi = torch.zeros(2, dtype=torch.int32)
    rc = pa.lib().pa_v2_plan(ip.data_ptr(), lp.data_ptr(), fp.data_ptr(), None, 1, 16, 8, 8, 128, pa.PA_F16,
                             10 ** 6, 0, ri.data_ptr(), ri.data_ptr(), 2, oi.data_ptr(), ctypes.byref(st))
    assert rc == pa.PA_ECAPACITY and st.num_chunks == 10


def test_plan_matches_predicate():
    b = W.sliding_window_batch()
    p = pa.pa_v2_plan(b.indptr, b.last_page_len, b.first_page_offset, 16, 32, 8, 128, pa.PA_BF16, 640)
    assert pa.pa_v2_plan_matches(p, b.indptr, b.last_page_len, b.first_page_offset)
    # one more token inside the last page: same pages, the plan still holds
    lpl = b.last_page_len.clone()
    r = int(torch.nonzero(lpl < 16)[0])
    lpl[r] += 1
    assert pa.pa_v2_plan_matches(p, b.indptr, lpl, b.first_page_offset)
    # a request crossing a page boundary: the plan must be rebuilt
    ip = b.indptr.clone()
    ip[r + 1:] += 1
    lpl2 = b.last_page_len.clone()
    lpl2[r] = 1
    assert not pa.pa_v2_plan_matches(p, ip, lpl2, b.first_page_offset)
    # invalid geometry never matches
    bad = b.last_page_len.clone()
    bad[0] = 0
    assert not pa.pa_v2_plan_matches(p, b.indptr, bad, b.first_page_offset)


def test_host_io_layout_sizes():
    b = W.tiny_csr()
    plan = pa.pa_v2_plan(b.indptr, b.last_page_len, b.first_page_offset, b.page_size, b.num_qo_heads,
                         b.num_kv_heads, b.head_dim, pa.PA_F32, 8, b.ppc_override, b.seq_lens)
    i, o, io = pa.pa_v2_host_io_layout(plan)
    words = b.q.numel() + b.indices.numel() + (b.batch + 1) + 2 * b.batch
    assert i == -(-words * 4 // 16) * 16 + 16 and i % 16 == 0
    assert o == 16 + b.q.numel() * 4 + b.batch * b.num_qo_heads * 4
    assert io == i - 16 + o


def _ctas(pages, size, per):
    return sum(max(1, -(-p // size)) for p in pages) * per


@pytest.mark.parametrize("seed", range(6))
def test_wave_fit_is_the_smallest_size_that_fits(seed):
    """Brute force over every chunk size: the result fits the wave and the size one below does not (or the
    result is the one-chunk-per-request size when nothing fits); it agrees with the Python helper."""
    import random
    from paged_attention_decode_gb300 import cascade as C
    rng = random.Random(seed)
    pages = [rng.choice([0, 1, 7, 64, 113, 2048, rng.randint(0, 3000)]) for _ in range(rng.randint(1, 9))]
    indptr = [0]
    for p in pages:
        indptr.append(indptr[-1] + p)
    for per, wave in ((1, 152), (8, 152), (4, 144), (16, 20), (3, 7)):
        got = pa.pa_v2_wave_fit_pages_per_chunk(indptr, per, wave)
        longest = max([1] + pages)
        if _ctas(pages, longest, per) > wave:
            assert got == longest
        else:
            assert _ctas(pages, got, per) <= wave
            assert got == 1 or _ctas(pages, got - 1, per) > wave
            assert got == min(s for s in range(1, longest + 1) if _ctas(pages, s, per) <= wave)
        assert got == C.fit_pages_per_chunk(pages, per, wave)


def test_wave_fit_on_the_sparse_shape_and_bad_arguments():
    # 16 requests of 2048 single-row pages, 1 KV head: the plan's search takes 227 pages (160 CTAs);
    # one wave of 152 holds 9 chunks per request (144 CTAs) at 228 pages
    indptr = [2048 * r for r in range(17)]
    assert pa.pa_v2_wave_fit_pages_per_chunk(indptr, 1, 152) == 228
    with pytest.raises(pa.PaError):
        pa.pa_v2_wave_fit_pages_per_chunk([0, 5], 0, 152)
    with pytest.raises(pa.PaError):
        pa.pa_v2_wave_fit_pages_per_chunk([1, 5], 1, 152)


def _stages(size, ps):
    return -(-size // (16 // ps)) if ps <= 16 else size * (ps // 16)


@pytest.mark.parametrize("seed", range(6))
def test_balanced_size_brute_force(seed):
    """Brute force: the result keeps the given size's chunk count, gives a stage count that is a multiple of
    8 (the tensor-core kernel's warps), and no larger size up to the given one does both; when no size
    does, the given size comes back."""
    import random
    rng = random.Random(100 + seed)
    pages = [rng.choice([0, 1, 5, 113, 2048, rng.randint(0, 3000)]) for _ in range(rng.randint(1, 6))]
    indptr = [0]
    for p in pages:
        indptr.append(indptr[-1] + p)
    for ps in (1, 2, 4, 8, 16, 32, 64):
        for ppc in sorted({1, 7, 8, 57, 113, 228, rng.randint(1, 3000)}):
            got = pa.pa_v2_balanced_pages_per_chunk(indptr, ps, ppc)
            want = _ctas(pages, ppc, 1)
            ok = [s for s in range(1, ppc + 1) if _stages(s, ps) % 8 == 0 and _ctas(pages, s, 1) == want]
            assert got == (max(ok) if ok else ppc), (pages, ps, ppc)


def test_balanced_size_on_the_32k_decode_and_bad_arguments():
    # 2048 pages of 16 rows: the plan's 113 pages per chunk make 19 chunks with 113 stages each (one warp
    # of 8 takes 15); 112 keeps 19 chunks at 14 stages per warp
    assert pa.pa_v2_balanced_pages_per_chunk([0, 2048], 16, 113) == 112
    assert pa.pa_v2_balanced_pages_per_chunk([0, 2048], 16, 112) == 112
    # 16 requests of 2048 one-row pages at 228 pages (15 stages of 16 pages): 8 stages would need 9 -> 16
    # chunks per request, so the size stays
    assert pa.pa_v2_balanced_pages_per_chunk([2048 * r for r in range(17)], 1, 228) == 228
    # 64-row pages: 4 stages per page, any even size balances
    assert pa.pa_v2_balanced_pages_per_chunk([0, 1000], 64, 101) == 100
    # page sizes above 16 that are not multiples of 16 are left alone
    assert pa.pa_v2_balanced_pages_per_chunk([0, 1000], 24, 101) == 101
    for bad in (([0, 5], 0, 3), ([0, 5], 16, 0), ([1, 5], 16, 3), ([0, 5, 4], 16, 3)):
        with pytest.raises(pa.PaError):
            pa.pa_v2_balanced_pages_per_chunk(*bad)


def test_host_graph_rejects_bad_arguments_before_any_cuda_call():
    import ctypes
    L = pa.lib()
    g = ctypes.c_void_p()
    args = [None] * 6 + [pa.PA_F16, 1, None, None, None, 0.1, None, None]
    assert L.pa_v2_host_graph_create(None, *args[1:], ctypes.byref(g)) == pa.PA_EINVAL
    assert L.pa_v2_host_graph_create(None, *args[1:], None) == pa.PA_EINVAL
    assert not g.value
    assert L.pa_v2_host_graph_run(None, None) == pa.PA_EINVAL
    L.pa_v2_host_graph_destroy(None)  # a no-op


def test_decode_and_merge_reject_bad_arguments_before_any_cuda_call():
    """Host-side validation of pa_v2_decode_partial / pa_v2_decode / pa_merge_states: every case below returns
    before a tensor map is encoded or a kernel launched (no device is needed), including the pool-row limit
    (num_pages * page_size must stay below 2^31) and a plan with no chunks (nothing to launch)."""
    import ctypes
    import math
    L = pa.lib()
    b = W.make_batch("args", [100, 40], [0, 3], 16, 8, 2, 128, torch.float16, seed=3)
    plan = pa.pa_v2_plan(b.indptr, b.last_page_len, b.first_page_offset, 16, 8, 2, 128, pa.PA_F16, 16)
    A = 1 << 20                                     # fake 16-byte-aligned addresses: never dereferenced

    def partial(s=None, q=A, dtype=pa.PA_F16, num_pages=64, num_indices=None, scale=0.1, v_out=A):
        s = plan.struct if s is None else s
        n = plan.num_indices if num_indices is None else num_indices
        return L.pa_v2_decode_partial(ctypes.byref(s) if s is not False else None, q, A, A, dtype, num_pages, A, n,
                                      A, A, A, A, A, scale, v_out, A, None, None)

    def mutated(**kw):
        s = pa.PlanStruct.from_buffer_copy(plan.struct)
        for k, v in kw.items():
            setattr(s, k, v)
        return s

    assert partial(s=False) == pa.PA_EINVAL
    assert partial(q=None) == pa.PA_EINVAL
    assert partial(q=A + 4) == pa.PA_EINVAL         # misaligned q
    assert partial(v_out=A + 8) == pa.PA_EINVAL     # misaligned workspace
    assert partial(dtype=pa.PA_BF16) == pa.PA_EINVAL
    assert partial(num_pages=0) == pa.PA_EINVAL
    assert partial(num_indices=plan.num_indices - 1) == pa.PA_EINVAL
    for bad in (math.inf, math.nan):
        assert partial(scale=bad) == pa.PA_EINVAL
    assert partial(num_pages=(1 << 31) // 16) == pa.PA_EUNSUPPORTED      # 2^31 pool rows
    assert partial(s=mutated(q_heads_per_cta=3)) == pa.PA_EINVAL
    assert partial(s=mutated(head_dim=96)) == pa.PA_EUNSUPPORTED
    assert partial(s=mutated(stack_members=0)) == pa.PA_EINVAL
    assert partial(s=mutated(num_chunks=0)) == pa.PA_OK                 # nothing to launch
    # the fused entry point: the same checks plus its merge arguments
    assert L.pa_v2_decode(ctypes.byref(plan.struct), A, A, A, pa.PA_F16, 64, A, plan.num_indices, A, A, A, A, A,
                          None, 0.1, A, A, A, A, A, None, None, None, None) == pa.PA_EINVAL   # no o_indptr
    # the merge
    assert L.pa_merge_states(A, A, A, 2, 5, 0, 128, A, A, None, None) == pa.PA_EINVAL     # no heads
    assert L.pa_merge_states(A, A, A, -1, 5, 8, 128, A, A, None, None) == pa.PA_EINVAL
    assert L.pa_merge_states(A + 4, A, A, 2, 5, 8, 128, A, A, None, None) == pa.PA_EINVAL  # misaligned v_in
    assert L.pa_merge_states(A, A, None, 2, 5, 8, 128, A, A, None, None) == pa.PA_EINVAL   # no o_indptr
    assert L.pa_merge_states(A, A, A, 0, 5, 8, 128, A, A, None, None) == pa.PA_OK          # no rows: no launch
