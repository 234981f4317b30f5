"""Pins of the f64 oracle against what the pages and mathematics fix (CPU only).

Each test checks the oracle against something other than itself: values worked
by hand from the pages (tests/golden/), library routines (numpy/torch element
decoding, torch scaled_dot_product_attention and logsumexp in f64), closed
forms, invariants the pages state (chunk-size invariance, merge associativity
and commutativity, cascade == flat) and brute force on tiny inputs.
"""
import math
import os
import random

import numpy as np
import pytest
import torch

import oracle
from paged_attention_decode_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TIGHT = 1e-12


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


# ---------------------------------------------------------------------------
# element decoding (IEEE binary16, bfloat16) against the libraries' conversions
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_element_decoding_every_bit_pattern(dtype):
    bits = torch.arange(0, 65536, dtype=torch.int32).to(torch.int16)
    vals = bits.view(dtype)
    ours = oracle.decode_elements(vals)
    ref = vals.double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_element_decoding_f32():
    v = torch.randn(1000, generator=torch.Generator().manual_seed(5))
    assert np.array_equal(oracle.decode_elements(v), v.double().numpy())


# ---------------------------------------------------------------------------
# CSR geometry
# ---------------------------------------------------------------------------

def test_geometry_golden_rows():
    for row in _read_golden("csr_geometry.txt"):
        lhs, rhs = row.split("->")
        ps, L, fpo = map(int, lhs.split())
        pages, lpl = map(int, rhs.split())
        assert W.page_geometry(L, fpo, ps) == (pages, lpl), row
        indptr = [0, pages]
        assert oracle.seq_lens(indptr, [lpl], [fpo if L else 0], ps) == [L], row
        assert oracle.validate_geometry(indptr, [lpl], [fpo if L else 0], ps,
                                        expect_seq_lens=[L]) == oracle.GEOM_OK, row


def test_exactly_full_final_page_is_page_size_not_zero():
    for ps in (1, 4, 16, 64):
        for pages in (1, 2, 7):
            assert W.page_geometry(pages * ps, 0, ps) == (pages, ps)
    assert oracle.validate_geometry([0, 2], [0], [0], 16) == oracle.GEOM_LAST_PAGE_LEN


def test_geometry_identity_on_workloads():
    for b in (W.tiny_csr(), W.sliding_window_batch(), W.cascade_mixed_batch(),
              W.sparse_token_exact(cap=4096, selected=64, heads=2),
              W.cascade_shared_prefix(prefix_tokens=256, suffix_range=(3, 40)).flat):
        assert oracle.validate_geometry(b.indptr, b.last_page_len, b.first_page_offset, b.page_size,
                                        b.indices, b.num_pages, b.seq_lens) == oracle.GEOM_OK, b.name


def test_tiny_workload_shape():
    b = W.tiny_csr()
    assert b.indptr.tolist() == [0, 4, 7]
    assert b.last_page_len.tolist() == [1, 1]
    assert b.first_page_offset.tolist() == [0, 2]
    assert b.num_pages == 16 and len(set(b.indices.tolist())) == 7


def test_sliding_window_workload_shape():
    b = W.sliding_window_batch()
    fpo = b.first_page_offset.tolist()
    assert b.seq_lens[:2] == [4096, 4096] and all(1 <= f <= 15 for f in fpo[:2])
    assert fpo[2:] == [0, 0] and all(1024 <= s <= 16384 for s in b.seq_lens[2:])
    # a 4096-token window starting mid-page spans 257 pages, the last holding fpo entries
    assert (b.indptr[1] - b.indptr[0]).item() == 257
    assert b.last_page_len[0].item() == fpo[0]


def _mutations(b):
    """(description, indptr, lpl, fpo, indices, expected code) for every rejection path."""
    ip = b.indptr.tolist()
    lp = b.last_page_len.tolist()
    fp = b.first_page_offset.tolist()
    idx = b.indices.tolist()
    ps = b.page_size
    out = []
    nonempty = [r for r in range(len(lp)) if ip[r + 1] > ip[r]]
    if not nonempty:
        return out
    r = nonempty[0]
    out.append(("indptr0", [1] + ip[1:], lp, fp, idx, oracle.GEOM_INDPTR0))
    bad = list(ip)
    bad[r + 1] = bad[r] - 1
    out.append(("order", bad, lp, fp, idx, oracle.GEOM_INDPTR_ORDER))
    out.append(("lpl0", ip, lp[:r] + [0] + lp[r + 1:], fp, idx, oracle.GEOM_LAST_PAGE_LEN))
    out.append(("lplbig", ip, lp[:r] + [ps + 1] + lp[r + 1:], fp, idx, oracle.GEOM_LAST_PAGE_LEN))
    out.append(("fpo", ip, lp, fp[:r] + [ps] + fp[r + 1:], idx, oracle.GEOM_FIRST_OFFSET))
    out.append(("fponeg", ip, lp, fp[:r] + [-1] + fp[r + 1:], idx, oracle.GEOM_FIRST_OFFSET))
    bad_idx = list(idx)
    bad_idx[ip[r]] = b.num_pages
    out.append(("pageid", ip, lp, fp, bad_idx, oracle.GEOM_PAGE_ID))
    bad_idx = list(idx)
    bad_idx[ip[r]] = -1
    out.append(("pageidneg", ip, lp, fp, bad_idx, oracle.GEOM_PAGE_ID))
    return out


def test_geometry_randomized_sweep_500():
    rng = random.Random(1234)
    for case in range(500):
        ps = rng.choice([1, 2, 3, 4, 5, 8, 12, 16, 17, 32, 64])
        B = rng.randint(1, 5)
        lens = [rng.choice([0, 1, rng.randint(1, 200), ps, 3 * ps]) for _ in range(B)]
        fpos = [rng.randrange(ps) if L else 0 for L in lens]
        b = W.make_batch(f"g{case}", lens, fpos, ps, num_qo_heads=1, num_kv_heads=1, head_dim=4,
                         dtype=torch.float32, seed=case)
        assert oracle.seq_lens(b.indptr, b.last_page_len, b.first_page_offset, ps) == lens
        assert oracle.validate_geometry(b.indptr, b.last_page_len, b.first_page_offset, ps, b.indices,
                                        b.num_pages, lens) == oracle.GEOM_OK
        wrong = list(lens)
        wrong[0] += 1
        assert oracle.validate_geometry(b.indptr, b.last_page_len, b.first_page_offset, ps,
                                        expect_seq_lens=wrong) == oracle.GEOM_IDENTITY
        for name, ip, lp, fp, idx, code in _mutations(b):
            got = oracle.validate_geometry(ip, lp, fp, ps, idx, b.num_pages)
            assert got == code, (case, name, got, code)


def test_geometry_single_page_window_and_empty_request():
    # one page whose window starts at or after its last valid entry has no visible token
    assert oracle.validate_geometry([0, 1], [3], [3], 16) == oracle.GEOM_SINGLE_PAGE
    # a request with no pages must report last_page_len = first_page_offset = 0
    assert oracle.validate_geometry([0, 0], [1], [0], 16) == oracle.GEOM_EMPTY_REQUEST
    assert oracle.validate_geometry([0, 0], [0], [0], 16) == oracle.GEOM_OK
    assert oracle.validate_geometry([0, 1], [1], [0], 0) == oracle.GEOM_BAD_ARGS


# ---------------------------------------------------------------------------
# page resolution against the scatter that built the pool
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("ps", [1, 3, 4, 16])
@pytest.mark.parametrize("order", ["shuffled", "reversed"])
def test_resolution_inverts_the_scatter(ps, order):
    g = torch.Generator().manual_seed(ps)
    lens, fpos = [9, 1, 0, 23], [0, ps - 1, 0, min(2, ps - 1)]
    dk = [torch.randn(L, 2, 4, generator=g) for L in lens]
    dv = [torch.randn(L, 2, 4, generator=g) for L in lens]
    b = W.scatter_dense("scatter", dk, dv, fpos, ps, num_qo_heads=2, seed=ps, order=order)
    flat_k = b.k_pool.reshape(-1, 2, 4)
    touched = set()
    for r, L in enumerate(lens):
        rows = oracle.resolve_rows(b.indices, b.indptr, b.first_page_offset, ps, r, L)
        assert torch.equal(flat_k[rows], dk[r]), (r, rows)
        touched.update(rows)
    untouched = [i for i in range(flat_k.shape[0]) if i not in touched]
    assert torch.isnan(flat_k[untouched]).all()


# ---------------------------------------------------------------------------
# attention against the dense library routine (brute force on tiny inputs)
# ---------------------------------------------------------------------------

def _dense_reference(q, dk, dv, scale):
    """torch SDPA and logsumexp in f64 on dense per-request sequences; GQA by head repetition."""
    B, Hq, D = q.shape
    outs, lses = [], []
    for r in range(B):
        K, V = dk[r].double(), dv[r].double()            # [L, Hkv, D]
        L, Hkv, _ = K.shape
        G = Hq // Hkv
        if L == 0:
            outs.append(torch.zeros(Hq, D, dtype=torch.float64))
            lses.append(torch.full((Hq,), -math.inf, dtype=torch.float64))
            continue
        Kh = K.permute(1, 0, 2).repeat_interleave(G, dim=0)   # [Hq, L, D]
        Vh = V.permute(1, 0, 2).repeat_interleave(G, dim=0)
        qh = q[r].double().unsqueeze(1)                       # [Hq, 1, D]
        o = torch.nn.functional.scaled_dot_product_attention(qh, Kh, Vh, scale=scale)
        s = torch.matmul(qh, Kh.transpose(1, 2)).squeeze(1) * scale
        outs.append(o.squeeze(1))
        lses.append(torch.logsumexp(s, dim=-1) / math.log(2.0))
    return torch.stack(outs).numpy(), torch.stack(lses).numpy()


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16, torch.bfloat16])
@pytest.mark.parametrize("G", [1, 3, 4])
def test_attention_matches_dense_sdpa(dtype, G):
    g = torch.Generator().manual_seed(G * 7)
    Hkv, D, ps = 2, 16, 4
    lens, fpos = [9, 1, 17, 0, 4], [0, 3, 1, 0, 2]
    dk = [torch.randn(L, Hkv, D, generator=g).to(dtype) for L in lens]
    dv = [torch.randn(L, Hkv, D, generator=g).to(dtype) for L in lens]
    b = W.scatter_dense("dense", dk, dv, fpos, ps, num_qo_heads=Hkv * G, seed=G, dtype=dtype)
    out, lse = oracle.attention(b.q, b.k_pool, b.v_pool, b.indices, b.indptr, b.last_page_len,
                                b.first_page_offset, b.scale)
    ref_o, ref_l = _dense_reference(b.q, dk, dv, b.scale)
    np.testing.assert_allclose(out, ref_o, rtol=0, atol=TIGHT)
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], ref_l[fin], rtol=0, atol=TIGHT)
    assert np.all(out[3] == 0) and np.all(lse[3] == -np.inf)   # the empty request


def test_attention_golden_hand_example():
    rows = _read_golden("attention_closed_form.txt")
    k = torch.full((3, 2, 1, 2), float("nan"), dtype=torch.float64)
    v = torch.full((3, 2, 1, 2), float("nan"), dtype=torch.float64)
    for row in rows[:2]:
        page, entry, k0, k1, v0, v1 = map(float, row.split())
        k[int(page), int(entry), 0] = torch.tensor([k0, k1])
        v[int(page), int(entry), 0] = torch.tensor([v0, v1])
    exp = list(map(float, rows[2].split()))
    q = torch.tensor([[[math.log(3.0), 0.0]]], dtype=torch.float32)
    out, lse = oracle.attention(q, k.float(), v.float(), [2, 0], [0, 2], [1], [1], 1.0)
    # q was rounded to f32, so ln 3 carries a 2^-24 relative error
    np.testing.assert_allclose(out[0, 0], exp[:2], rtol=0, atol=1e-7)
    np.testing.assert_allclose(lse[0, 0], exp[2], rtol=0, atol=1e-7)


def test_closed_forms():
    g = torch.Generator().manual_seed(3)
    b = W.make_batch("cf", [1, 40, 40], [5, 3, 0], page_size=8, num_qo_heads=4, num_kv_heads=2,
                     head_dim=32, dtype=torch.float32, seed=11)
    # seq_len 1: output is that token's V exactly, lse2 = s0 * log2(e)
    out, lse = oracle.attention(b.q, b.k_pool, b.v_pool, b.indices, b.indptr, b.last_page_len,
                                b.first_page_offset, b.scale)
    row = oracle.resolve_rows(b.indices, b.indptr, b.first_page_offset, 8, 0, 1)[0]
    kf = b.k_pool.reshape(-1, 2, 32).double()
    vf = b.v_pool.reshape(-1, 2, 32).double()
    for h in range(4):
        assert np.array_equal(out[0, h], vf[row, h // 2].numpy())
        s0 = b.scale * float(b.q[0, h].double() @ kf[row, h // 2])
        assert abs(lse[0, h] - s0 / math.log(2.0)) < TIGHT
    # constant V rows: output equals that constant for any q
    v_const = torch.zeros_like(b.v_pool) + torch.linspace(-2, 2, 32)
    out, _ = oracle.attention(b.q, b.k_pool, v_const, b.indices, b.indptr, b.last_page_len,
                              b.first_page_offset, b.scale)
    np.testing.assert_allclose(out, np.broadcast_to(torch.linspace(-2, 2, 32).double().numpy(), out.shape),
                               rtol=0, atol=TIGHT)
    # q = 0: uniform softmax, output is the mean of V, lse2 = log2(seq_len)
    out, lse = oracle.attention(torch.zeros_like(b.q), b.k_pool, b.v_pool, b.indices, b.indptr,
                                b.last_page_len, b.first_page_offset, b.scale)
    for r, L in enumerate(b.seq_lens):
        rows = oracle.resolve_rows(b.indices, b.indptr, b.first_page_offset, 8, r, L)
        for h in range(4):
            np.testing.assert_allclose(out[r, h], vf[rows, h // 2].mean(0).numpy(), rtol=0, atol=TIGHT)
            assert abs(lse[r, h] - math.log2(L)) < TIGHT


def test_page_table_sensitivity():
    """Shuffled physical pages: a reading that ignored ``indices`` would get another answer."""
    b = W.make_batch("sens", [50, 33], [0, 7], page_size=8, num_qo_heads=2, num_kv_heads=1,
                     head_dim=16, dtype=torch.float16, seed=21, order="shuffled")
    out, _ = oracle.attention(b.q, b.k_pool, b.v_pool, b.indices, b.indptr, b.last_page_len,
                              b.first_page_offset, b.scale)
    ident = torch.arange(len(b.indices), dtype=torch.int32)
    out_id, _ = oracle.attention(b.q, b.k_pool, b.v_pool, ident, b.indptr, b.last_page_len,
                                 b.first_page_offset, b.scale)
    assert np.abs(out - out_id).max() > 0.05


def test_sparse_selection_set_equality():
    """Page size 1 over a dense [B, H, Cap, D] cache: the attended rows are exactly the selected
    positions of request r = b * H + h (sparse-paged-decode.md, issue #904)."""
    b = W.sparse_token_exact(cap=4096, selected=64, heads=2, batch=2)
    cap = b.meta["cap"]
    for r, pos in enumerate(b.meta["positions"]):
        rows = oracle.resolve_rows(b.indices, b.indptr, b.first_page_offset, 1, r, 64)
        assert sorted(rows) == sorted((r * cap + pos).tolist())
        assert len(set(rows)) == 64


# ---------------------------------------------------------------------------
# chunked partials and the merge
# ---------------------------------------------------------------------------

def _ragged_batch(dtype=torch.float32, seed=31):
    """Ragged requests (empty, one token, mid-page starts, final pages of 8, 1 and 7 entries) in a
    pool whose every entry outside the sequences is NaN, so a read past any range shows up."""
    g = torch.Generator().manual_seed(seed)
    lens, fpos = [37, 0, 1, 64, 24, 9], [3, 0, 0, 0, 7, 0]
    dk = [torch.randn(L, 2, 16, generator=g) for L in lens]
    dv = [torch.randn(L, 2, 16, generator=g) for L in lens]
    return W.scatter_dense("ragged", dk, dv, fpos, 8, num_qo_heads=6, seed=seed, dtype=dtype)


def test_chunk_size_invariance_every_ppc():
    b = _ragged_batch()
    ref_o, ref_l = oracle.attention(b.q, b.k_pool, b.v_pool, b.indices, b.indptr, b.last_page_len,
                                    b.first_page_offset, b.scale)
    hi = int((b.indptr[1:] - b.indptr[:-1]).max())
    for ppc in range(1, hi + 2):
        p = oracle.plan(b.indptr, b.num_kv_heads, 1, 1, ppc_override=ppc)
        v, l = oracle.partials(b.q, b.k_pool, b.v_pool, b.indices, b.indptr, b.last_page_len,
                               b.first_page_offset, b.scale, ppc, p.request_indices, p.kv_tile_indices)
        o, lse = oracle.merge(v, l, p.o_indptr)
        np.testing.assert_allclose(o, ref_o, rtol=0, atol=TIGHT)
        fin = np.isfinite(ref_l)
        assert np.array_equal(np.isfinite(lse), fin)
        np.testing.assert_allclose(lse[fin], ref_l[fin], rtol=0, atol=TIGHT)


def test_partial_of_empty_chunk_is_zero_and_minus_inf():
    b = _ragged_batch()
    p = oracle.plan(b.indptr, b.num_kv_heads, 1, 1, ppc_override=2)
    v, l = oracle.partials(b.q, b.k_pool, b.v_pool, b.indices, b.indptr, b.last_page_len,
                           b.first_page_offset, b.scale, 2, p.request_indices, p.kv_tile_indices)
    empty = [c for c, r in enumerate(p.request_indices) if r == 1]
    assert len(empty) == 1
    assert np.all(v[empty] == 0) and np.all(l[empty] == -np.inf)


def _random_states(N, H, D, seed, neg_inf_rows=()):
    g = np.random.default_rng(seed)
    v = g.standard_normal((N, H, D))
    l = g.uniform(-20, 20, (N, H))
    for i in neg_inf_rows:
        v[i] = 0.0
        l[i] = -np.inf
    return v, l


def test_merge_commutative_and_associative():
    v, l = _random_states(9, 3, 8, 1)
    full_o, full_l = oracle.merge(v, l, [0, 9])
    perm = np.random.default_rng(2).permutation(9)
    po, pl = oracle.merge(v[perm], l[perm], [0, 9])
    np.testing.assert_allclose(po, full_o, rtol=0, atol=TIGHT)
    np.testing.assert_allclose(pl, full_l, rtol=0, atol=TIGHT)
    for cut in ([0, 4, 9], [0, 1, 9], [0, 3, 6, 9], [0, 8, 9]):
        mo, ml = oracle.merge(v, l, cut)
        ro, rl = oracle.merge(mo, ml, [0, len(cut) - 1])
        np.testing.assert_allclose(ro, full_o, rtol=0, atol=TIGHT)
        np.testing.assert_allclose(rl, full_l, rtol=0, atol=TIGHT)


def test_merge_single_row_is_identity_and_empty_rows():
    v, l = _random_states(5, 2, 4, 3, neg_inf_rows=(2, 3))
    o, lse = oracle.merge(v, l, [0, 1, 2, 4, 5])
    assert np.array_equal(o[0], v[0]) and np.array_equal(lse[0], l[0])
    assert np.array_equal(o[1], v[1]) and np.array_equal(lse[1], l[1])
    assert np.all(o[2] == 0) and np.all(lse[2] == -np.inf)        # all-empty group
    # a -inf member contributes nothing
    o2, l2 = oracle.merge(v[[0, 2]], l[[0, 2]], [0, 2])
    assert np.array_equal(o2[0], v[0]) and np.array_equal(l2[0], l[0])


def test_merge_of_disjoint_ranges_is_the_whole_range():
    """Two states over a partition of the key range merge to the attention over the whole range
    (issue #898, design piece 3)."""
    b = W.make_batch("two", [40], [0], page_size=4, num_qo_heads=2, num_kv_heads=1, head_dim=8,
                     dtype=torch.float32, seed=77)
    ref_o, ref_l = oracle.attention(b.q, b.k_pool, b.v_pool, b.indices, b.indptr, b.last_page_len,
                                    b.first_page_offset, b.scale)
    v, l = oracle.partials(b.q, b.k_pool, b.v_pool, b.indices, b.indptr, b.last_page_len,
                           b.first_page_offset, b.scale, 7, [0, 0], [0, 1])
    m = np.maximum(l[0], l[1])
    w0, w1 = 2.0 ** (l[0] - m), 2.0 ** (l[1] - m)
    by_hand = (w0[:, None] * v[0] + w1[:, None] * v[1]) / (w0 + w1)[:, None]
    np.testing.assert_allclose(by_hand, ref_o[0], rtol=0, atol=TIGHT)
    np.testing.assert_allclose(np.log2(w0 + w1) + m, ref_l[0], rtol=0, atol=TIGHT)
    o, lse = oracle.merge(v, l, [0, 2])
    np.testing.assert_allclose(o[0], ref_o[0], rtol=0, atol=TIGHT)


# ---------------------------------------------------------------------------
# cascade
# ---------------------------------------------------------------------------

def test_mixed_batch_detection_finds_the_planted_group():
    b = W.cascade_mixed_batch()
    assert oracle.cascade_detect_ref(b.indptr, b.indices, b.first_page_offset) == \
        (b.meta["members"], b.meta["shared_pages"])


def test_cascade_equals_flat_and_member_major_is_wrong():
    cb = W.cascade_shared_prefix(prefix_tokens=128, suffix_range=(5, 40), num_qo_heads=8, num_kv_heads=2,
                                 head_dim=16, page_size=16)
    f = cb.flat
    flat_o, flat_l = oracle.attention(f.q, f.k_pool, f.v_pool, f.indices, f.indptr, f.last_page_len,
                                      f.first_page_offset, f.scale)
    co, cl = oracle.cascade_ref(f.q, f.k_pool, f.v_pool, cb.prefix_indices, cb.suffix_indices,
                                cb.suffix_indptr, cb.suffix_last_page_len, f.scale)
    np.testing.assert_allclose(co, flat_o, rtol=0, atol=TIGHT)
    np.testing.assert_allclose(cl, flat_l, rtol=0, atol=TIGHT)
    # negative control: stacking member-major maps query heads to the wrong KV head
    M, Hq, D = f.q.shape
    q_wrong = f.q.reshape(1, M * Hq, D)
    npre = len(cb.prefix_indices)
    o0, _ = oracle.attention(q_wrong, f.k_pool, f.v_pool, cb.prefix_indices, [0, npre], [16], [0], f.scale)
    o_right, _ = oracle.attention(
        f.q.reshape(M, 2, Hq // 2, D).permute(1, 0, 2, 3).reshape(1, M * Hq, D),
        f.k_pool, f.v_pool, cb.prefix_indices, [0, npre], [16], [0], f.scale)
    right = torch.from_numpy(o_right).reshape(2, M, Hq // 2, D).permute(1, 0, 2, 3).reshape(M, Hq, D)
    wrong = torch.from_numpy(o0).reshape(M, Hq, D)
    assert (right - wrong).abs().max() > 0.05


# ---------------------------------------------------------------------------
# plan
# ---------------------------------------------------------------------------

def test_plan_golden_examples():
    for row in _read_golden("plan_examples.txt"):
        lhs, rhs = row.split("->")
        name, pages, hkv, target, override = [x.strip() for x in lhs.split("|")]
        ppc, n, ri, ti, oi = [x.strip() for x in rhs.split("|")]
        pages = list(map(int, pages.split()))
        indptr = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
        p = oracle.plan(indptr, int(hkv), 1, int(target), int(override))
        assert p.pages_per_chunk == int(ppc), name
        assert p.num_chunks == int(n), name
        if ri != "*":
            assert p.request_indices.tolist() == list(map(int, ri.split())), name
            assert p.kv_tile_indices.tolist() == list(map(int, ti.split())), name
        assert p.o_indptr.tolist() == list(map(int, oi.split())), name


def _chunks(pages, ppc):
    return sum(max(1, -(-p // ppc)) for p in pages)


def test_plan_is_maximal_and_launchable_random():
    rng = random.Random(99)
    for case in range(300):
        B = rng.randint(1, 12)
        pages = [rng.choice([0, 1, rng.randint(1, 3000)]) for _ in range(B)]
        indptr = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
        hkv = rng.choice([1, 2, 8])
        qg = rng.choice([1, 2])
        target = rng.randint(1, 5000)
        maxc = rng.choice([65535, 500])
        hi = max(1, max(pages))
        if _chunks(pages, hi) > maxc:
            continue
        p = oracle.plan(indptr, hkv, qg, target, max_chunks=maxc)
        # floor: lo is the smallest launchable chunk size
        assert _chunks(pages, p.lo) <= maxc and (p.lo == 1 or _chunks(pages, p.lo - 1) > maxc)
        assert p.hi == hi and p.lo <= p.pages_per_chunk <= hi
        ctas = lambda c: _chunks(pages, c) * hkv * qg
        if ctas(p.lo) >= target:
            assert ctas(p.pages_per_chunk) >= target
            assert p.pages_per_chunk == hi or ctas(p.pages_per_chunk + 1) < target
        else:
            assert p.pages_per_chunk == p.lo
        # at least one chunk per request, request-major, tiles ascending
        assert p.num_chunks == _chunks(pages, p.pages_per_chunk)
        for r in range(B):
            rows = list(range(p.o_indptr[r], p.o_indptr[r + 1]))
            assert len(rows) == max(1, -(-pages[r] // p.pages_per_chunk))
            assert p.request_indices[rows].tolist() == [r] * len(rows)
            assert p.kv_tile_indices[rows].tolist() == list(range(len(rows)))


def test_plan_grid_floor_binds():
    pages = [40] * 4000        # ppc 1 would need 160000 chunks
    indptr = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
    p = oracle.plan(indptr, 8, 1, 10 ** 9)
    assert p.lo == 3 and p.pages_per_chunk == 3      # ceil(40/2)*4000 = 80000 > 65535, ceil(40/3)*4000 = 56000
