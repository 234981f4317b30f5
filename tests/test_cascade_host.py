"""Cascade detection and level split on the host (no GPU): the library against the oracle's rule."""
import random

import pytest
import torch

import oracle
from paged_attention_decode_gb300 import pa_v2 as pa


def _batch(rng, B, shared_groups):
    """Random page tables where some requests copy a leading run of pages from a donor."""
    tables, fpos = [], []
    next_id = 0
    for r in range(B):
        n = rng.randint(1, 60)
        pages = list(range(next_id, next_id + n))
        next_id += n
        if tables and rng.random() < shared_groups:
            donor = rng.choice(tables)
            k = rng.randint(1, len(donor))
            pages = donor[:k] + pages[:max(1, n - k)]
        tables.append(pages)
        fpos.append(rng.choice([0, 0, 0, rng.randint(1, 15)]))
    indptr = [0]
    for t in tables:
        indptr.append(indptr[-1] + len(t))
    indices = [p for t in tables for p in t]
    lpl = [rng.randint(max(1, f + 1) if len(t) == 1 else 1, 16) for t, f in zip(tables, fpos)]
    return indptr, indices, lpl, fpos


def test_detect_matches_the_oracle_rule_random():
    rng = random.Random(5)
    hits = 0
    for case in range(400):
        B = rng.randint(1, 12)
        indptr, indices, lpl, fpo = _batch(rng, B, 0.6)
        ms, mm = rng.choice([(1, 2), (4, 2), (16, 2), (3, 3)])
        ref_members, ref_shared = oracle.cascade_detect_ref(indptr, indices, fpo, ms, mm)
        flags, shared = pa.pa_v2_cascade_detect(indptr, indices, fpo, ms, mm)
        got = [r for r in range(B) if int(flags[r])]
        assert (got, shared) == (ref_members, ref_shared), (case, got, shared, ref_members, ref_shared)
        hits += bool(got)
    assert hits > 50


def test_detect_rules_by_hand():
    # three requests share pages 10..29; request 3 shares them too but starts mid-page; request 4 shares
    # only page 10 and 11
    t = [list(range(10, 30)) + [100 + i for i in range(5)],
         list(range(10, 30)) + [200],
         list(range(10, 30)) + [300, 301],
         list(range(10, 30)) + [400],
         [10, 11, 500]]
    fpo = [0, 0, 0, 3, 0]
    indptr = [0]
    for x in t:
        indptr.append(indptr[-1] + len(x))
    indices = [p for x in t for p in x]
    # the group keyed by page 10 is {0, 1, 2, 4}; request 4 caps the span at 2 pages
    assert oracle.cascade_detect_ref(indptr, indices, fpo, 1, 2) == ([0, 1, 2, 4], 2)
    flags, shared = pa.pa_v2_cascade_detect(indptr, indices, fpo, 1, 2)
    assert flags.tolist() == [1, 1, 1, 0, 1] and shared == 2
    # below the minimum span nothing qualifies
    assert pa.pa_v2_cascade_detect(indptr, indices, fpo, 16, 2)[1] == 0
    # a request whose span reaches its last page caps the span at pages - 1
    t2 = [list(range(10, 30)), list(range(10, 30)) + [7]]
    ip2 = [0, 20, 41]
    idx2 = t2[0] + t2[1]
    assert oracle.cascade_detect_ref(ip2, idx2, [0, 0], 1, 2) == ([0, 1], 19)
    assert pa.pa_v2_cascade_detect(ip2, idx2, [0, 0], 1, 2)[1] == 19


def test_detect_tie_goes_to_the_group_met_first():
    # two groups remove the same number of page reads: the one keyed by page 50 (requests 0, 2, 4, three
    # shared pages: 3 x 2 = 6) and the one keyed by page 10 (requests 1, 3, six shared pages: 6 x 1 = 6).
    # The pages name the larger saving the winner and say nothing of a tie; the reading taken is that the
    # group whose first member comes first in the batch wins.  Reordering the batch flips the winner.
    g50 = [[50, 51, 52, 60, 61], [50, 51, 52, 80], [50, 51, 52, 95]]
    g10 = [list(range(10, 16)) + [70], list(range(10, 16)) + [90, 91]]
    for tables, want in (([g50[0], g10[0], g50[1], g10[1], g50[2]], ([0, 2, 4], 3)),
                         ([g10[0], g50[0], g10[1], g50[1], g50[2]], ([0, 2], 6))):
        indptr = [0]
        for x in tables:
            indptr.append(indptr[-1] + len(x))
        indices = [p for x in tables for p in x]
        fpo = [0] * len(tables)
        assert oracle.cascade_detect_ref(indptr, indices, fpo, 1, 2) == want
        flags, shared = pa.pa_v2_cascade_detect(indptr, indices, fpo, 1, 2)
        assert ([r for r in range(len(tables)) if int(flags[r])], shared) == want


def test_split_rebuilds_the_flat_tables():
    rng = random.Random(9)
    for case in range(100):
        B = rng.randint(2, 10)
        indptr, indices, lpl, fpo = _batch(rng, B, 0.8)
        flags, shared = pa.pa_v2_cascade_detect(indptr, indices, fpo, 1, 2)
        if shared == 0:
            continue
        sp = pa.pa_v2_cascade_split(indptr, indices, lpl, fpo, flags, shared)
        members = [r for r in range(B) if int(flags[r])]
        assert sp["member_rows"].tolist() == members
        first = members[0]
        prefix = indices[indptr[first]:indptr[first] + shared]
        mi = sp["merge_indptr"].tolist()
        for r in range(B):
            l1 = sp["l1_indices"][sp["l1_indptr"][r]:sp["l1_indptr"][r + 1]].tolist()
            full = indices[indptr[r]:indptr[r + 1]]
            assert (prefix + l1 if flags[r] else l1) == full
            assert mi[r + 1] - mi[r] == (2 if flags[r] else 1)
            assert sp["l1_out_rows"][r] == mi[r + 1] - 1
        assert sp["l0_out_rows"].tolist() == [mi[r] for r in members]


def test_cascade_plan_by_hand():
    # 4 members share 512 pages; suffixes of 25, 94, 62 and 91 pages; one wave of 152 CTAs, 8 CTAs per chunk at
    # either level (Hkv 8, one q-group).  The common size: 47 pages make 11 + (1 + 2 + 2 + 2) = 18 chunks = 144
    # CTAs; 46 pages would make 12 + (1 + 3 + 2 + 2) = 20 = 160.  Level 1 keeps 47 (7 chunks, 56 CTAs); level 0
    # takes the other 96 CTAs: 12 chunks, ceil(512 / 12) = 43 pages (11 x 43 + 39)
    c = pa.pa_v2_cascade_plan(4, 512, [0, 25, 119, 181, 272], [16, 4, 7, 16], [0, 0, 0, 0], 16, 32, 8, 128,
                              pa.PA_F16, 152)
    assert (c.level0.pages_per_chunk, c.level0.num_chunks, c.level1.num_chunks) == (43, 12, 7)
    assert c.level1.pages_per_chunk == 47 and c.level0.total_ctas + c.level1.total_ctas == 152
    assert (c.level0.stack_members, c.level0.num_qo_heads, c.level0.batch) == (4, 128, 1)
    # merge input, request by request: 12 level-0 rows then the request's level-1 rows
    assert c.merge_indptr.tolist() == [0, 13, 27, 41, 55]
    assert c.l0_part_rows.tolist() == [0, 13, 27, 41]
    # level-1 chunk j of request r lands at l1_part_rows[r] + j: chunks 0 | 1, 2 | 3, 4 | 5, 6
    assert c.l1_part_rows.tolist() == [12, 24, 36, 48]


def test_cascade_plan_brute_force():
    """The chunk sizes and the merge layout against their definitions on random batches, members anywhere in
    the level-1 table: level 1 at the smallest common size whose CTAs over both levels fit the wave, level 0 at
    the smallest size whose chunks fit beside level 1's; each request's rows are its level-0 chunks (members)
    then its level-1 chunks; every row is written exactly once."""
    rng = random.Random(11)
    for _ in range(300):
        B = rng.randint(1, 7)
        M = rng.randint(1, B)
        mreq = rng.sample(range(B), M)
        Hkv = rng.choice([1, 2, 8])
        G = rng.choice([1, 2, 4])
        shared = rng.randint(1, 600)
        pages = [rng.randint(1, 300) for _ in range(B)]
        ip = [0]
        for n in pages:
            ip.append(ip[-1] + n)
        wave = rng.randint(1, 400)
        c = pa.pa_v2_cascade_plan(M, shared, ip, [16] * B, [0] * B, 16, Hkv * G, Hkv, 128, pa.PA_F16, wave,
                                  member_requests=mreq)
        hpc0 = min(M * G, 16)
        per0, per1 = Hkv * -(-(M * G) // hpc0), Hkv

        def ctas(k):
            return per0 * -(-shared // k) + per1 * sum(max(1, -(-p // k)) for p in pages)
        fits = [k for k in range(1, max(pages + [shared]) + 1) if ctas(k) <= wave]
        want = min(fits) if fits else max(pages + [shared])
        assert c.level1.pages_per_chunk == want
        want0 = want
        if fits:
            ctas1 = per1 * sum(max(1, -(-p // want)) for p in pages)
            want0 = min(k for k in range(1, want + 1) if per0 * -(-shared // k) + ctas1 <= wave)
            assert c.level0.total_ctas + c.level1.total_ctas <= wave
        assert c.level0.pages_per_chunk == want0, (want0, c.level0.pages_per_chunk)
        assert c.level0.num_chunks == -(-shared // want0)
        n0 = c.level0.num_chunks
        o1 = c.level1.o_indptr.tolist()
        rows = []
        mi = c.merge_indptr.tolist()
        for r in range(B):
            mine = []
            if r in mreq:
                base = int(c.l0_part_rows[mreq.index(r)])
                mine += [base + k for k in range(n0)]
            mine += [int(c.l1_part_rows[r]) + j for j in range(o1[r], o1[r + 1])]
            assert mine == list(range(mi[r], mi[r + 1])), (r, mine, mi)
            rows += mine
        assert rows == list(range(c.merge_rows))


def test_cascade_plan_rejects_bad_arguments():
    for args in ((0, 16), (2, 0), (3, 16)):          # no member, no shared page, more members than requests
        with pytest.raises(pa.PaError) as e:
            pa.pa_v2_cascade_plan(*args, [0, 3, 5], [16, 16], [0, 0], 16, 32, 8, 128, pa.PA_F16, 152)
        assert e.value.status == pa.PA_EINVAL
    with pytest.raises(pa.PaError):
        pa.pa_v2_cascade_plan(2, 16, [0, 3, 5], [16, 16], [0, 0], 16, 32, 8, 128, pa.PA_F16, 0)
    with pytest.raises(pa.PaError):                   # a member listed twice
        pa.pa_v2_cascade_plan(2, 16, [0, 3, 5], [16, 16], [0, 0], 16, 32, 8, 128, pa.PA_F16, 152,
                              member_requests=[1, 1])


def test_chunk_fit_helper():
    from paged_attention_decode_gb300 import cascade as C
    # smallest chunk size whose CTAs fit the budget, by brute force
    rng = random.Random(3)
    for _ in range(300):
        pages = [rng.randint(0, 300) for _ in range(rng.randint(1, 6))]
        per = rng.choice([1, 8, 16])
        budget = rng.randint(1, 400)
        ppc = C.fit_pages_per_chunk(pages, per, budget)
        fits = [k for k in range(1, max(pages + [1]) + 1) if C._chunks(pages, k) * per <= budget]
        assert ppc == (min(fits) if fits else max(pages + [1]))
