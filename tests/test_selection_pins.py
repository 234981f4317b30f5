"""Pins of the block-sparse selection oracle (sparse-paged-decode.md, issue #904): block ids -> token
rows for a token-exact page table, and the block-granular page table of a pool-backed cache.  CPU only.

Pinned against: rows worked by hand (tests/golden/selection_from_blocks.txt), set equality with a keep
mask built position by position (the page's own check: attended positions == the mask path's kept
columns, across context lengths including a partial final block), and masked dense attention computed
by torch's scaled_dot_product_attention in f64.
"""
import math
import os
import random

import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "selection_from_blocks.txt")


def _golden():
    cases = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, ids, rows = [x.strip() for x in line.split("|")]
        C, kv_len, S = map(int, head.split())
        sel = [[int(x) for x in part.split()] for part in ids.split(";")]
        exp = [[int(x) for x in part.split()] for part in rows.split(";")]
        cases.append((C, kv_len, S, sel, exp))
    return cases


@pytest.mark.parametrize("case", range(len(_golden())))
def test_rows_match_hand_worked_examples(case):
    C, kv_len, S, sel, exp = _golden()[case]
    ids = torch.tensor(sel, dtype=torch.int32).reshape(len(sel), -1)
    rows, per = oracle.selection_rows_ref(ids, C, kv_len, S)
    assert per == len(exp[0])
    assert rows.tolist() == [x for e in exp for x in e]


def _keep_mask(sel, C, kv_len):
    """The mask path: position t is kept when its block is selected or is the final block."""
    nb = -(-kv_len // C)
    return [t // C in set(sel) or t // C == nb - 1 for t in range(kv_len)]


@pytest.mark.parametrize("kv_len", [1024, 1000, 1153, 4096 + 37])
def test_attended_positions_equal_the_mask_paths_kept_columns(kv_len):
    rng = random.Random(kv_len)
    C, R, S = 64, 3, kv_len + 77
    nb = -(-kv_len // C)
    topk = min(5, nb - 1)
    sel = [rng.sample(range(nb - 1), topk) for _ in range(R)]
    rows, per = oracle.selection_rows_ref(torch.tensor(sel, dtype=torch.int32), C, kv_len, S)
    assert per == topk * C + (kv_len - (nb - 1) * C)        # a function of kv_len, not of the scores
    rows = rows.tolist()
    for r in range(R):
        mine = rows[r * per:(r + 1) * per]
        assert len(set(mine)) == per                           # no row twice
        kept = {t for t, k in enumerate(_keep_mask(sel[r], C, kv_len)) if k}
        assert {x - r * S for x in mine} == kept
        assert all(0 <= x - r * S < kv_len for x in mine)      # never past the live window


def test_out_of_range_block_ids_are_rejected():
    C, kv_len = 4, 10                                          # nb = 3: scored blocks 0 and 1
    for bad in (2, 3, -1):
        with pytest.raises(ValueError):
            oracle.selection_rows_ref(torch.tensor([[bad]]), C, kv_len, 16)


def test_sparse_csr_structure():
    ip, lpl, fpo = oracle.sparse_csr_ref(3, 7)
    assert ip.tolist() == [0, 7, 14, 21] and lpl.tolist() == [1, 1, 1] and fpo.tolist() == [0, 0, 0]
    assert oracle.seq_lens(ip, lpl, fpo, 1) == [7, 7, 7]


def _dense_masked_attention(q, k, v, keep, scale):
    """SDPA in f64 over the live window with the keep mask as an additive -inf bias."""
    bias = torch.where(torch.tensor(keep), 0.0, -math.inf).to(torch.float64)
    o = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], v[None], attn_mask=bias[None, None],
                                                         scale=scale)[0]
    s = (q @ k.T) * scale + bias
    return o, torch.logsumexp(s, dim=-1) / math.log(2.0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16])
def test_token_exact_selection_equals_masked_dense_attention(dtype):
    gen = torch.Generator().manual_seed(11)
    C, kv_len, topk, R, n_rep, D = 4, 37, 3, 4, 2, 16
    S = kv_len + 5                                             # reserved capacity > live length
    nb = -(-kv_len // C)
    k = torch.randn(R * S, 1, 1, D, generator=gen).to(dtype)
    v = torch.randn(R * S, 1, 1, D, generator=gen).to(dtype)
    q = torch.randn(R, n_rep, D, generator=gen)
    sel = [torch.randperm(nb - 1, generator=gen)[:topk].tolist() for _ in range(R)]
    rows, per = oracle.selection_rows_ref(torch.tensor(sel, dtype=torch.int32), C, kv_len, S)
    ip, lpl, fpo = oracle.sparse_csr_ref(R, per)
    scale = 1.0 / math.sqrt(D)
    out, lse = oracle.attention(q, k, v, rows, ip, lpl, fpo, scale)
    for r in range(R):
        kd = k[r * S:r * S + kv_len, 0, 0].double()
        vd = v[r * S:r * S + kv_len, 0, 0].double()
        o_ref, l_ref = _dense_masked_attention(q[r].double(), kd, vd, _keep_mask(sel[r], C, kv_len), scale)
        assert torch.allclose(torch.as_tensor(out[r]).double(), o_ref, atol=1e-12, rtol=0)
        assert torch.allclose(torch.as_tensor(lse[r]).double(), l_ref, atol=1e-12, rtol=0)


def test_block_granular_pages_equal_token_exact_rows():
    """Pool-backed cache: the same selection as whole pages of block_size rows gives the same attention."""
    gen = torch.Generator().manual_seed(12)
    C, kv_len, topk, R, n_rep, D = 8, 61, 4, 3, 2, 16
    nb = -(-kv_len // C)
    bpr = nb + 2                                               # pool pages per request
    k = torch.randn(R * bpr * C, 1, 1, D, generator=gen).half()
    v = torch.randn(R * bpr * C, 1, 1, D, generator=gen).half()
    q = torch.randn(R, n_rep, D, generator=gen)
    sel = torch.stack([torch.randperm(nb - 1, generator=gen)[:topk] for _ in range(R)]).to(torch.int32)
    rows, per = oracle.selection_rows_ref(sel, C, kv_len, bpr * C)
    ip, lpl, fpo = oracle.sparse_csr_ref(R, per)
    o1, l1 = oracle.attention(q, k, v, rows, ip, lpl, fpo, 0.25)
    pages, ip2, lpl2, fpo2 = oracle.selection_pages_ref(sel, C, kv_len, bpr)
    o2, l2 = oracle.attention(q, k.reshape(R * bpr, C, 1, D), v.reshape(R * bpr, C, 1, D), pages, ip2, lpl2, fpo2,
                              0.25)
    assert float(abs(torch.as_tensor(o1) - torch.as_tensor(o2)).max()) < 1e-12
    assert float(abs(torch.as_tensor(l1) - torch.as_tensor(l2)).max()) < 1e-12
    assert oracle.seq_lens(ip2, lpl2, fpo2, C) == [per] * R
