"""Pins of the second-K-stream oracle (sparse-paged-decode.md, the DSA paragraphs: score =
scale * (q . k[row] + q_extra . k_extra[row]), values from v[row]).  CPU only.

Pinned against: the pinned single-stream oracle when q_extra is zero; torch's scaled_dot_product_attention
in f64 on the concatenated rows (the page's own exactness argument for concat(kv_latent, k_pe)); closed
forms (one token; an extra term that dominates); the merge of per-chunk partials for every chunk size.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_attention_decode_gb300 import workloads as W


def _case(seed=0, B=3, Hq=8, Hkv=2, D=32, E=8, stride=40, ps=4, seq=(13, 7, 1), fpo=(0, 2, 3),
          dtype=torch.float16):
    gen = torch.Generator().manual_seed(seed)
    b = W.make_batch("x", list(seq), list(fpo), ps, Hq, Hkv, stride, dtype, seed=seed + 1)
    ke = torch.randn(b.k_pool.shape[0], ps, Hkv, E, generator=gen).to(dtype)
    q = torch.randn(B, Hq, D, generator=gen)
    qe = torch.randn(B, Hq, E, generator=gen)
    return b, q, qe, ke


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16, torch.float32])
def test_zero_extra_query_reduces_to_the_single_stream_oracle(dtype):
    b, q, qe, ke = _case(dtype=dtype)
    D = q.shape[2]
    o1, l1 = oracle.attention_extra(q, torch.zeros_like(qe), b.k_pool, ke, b.v_pool, D, b.indices, b.indptr,
                                    b.last_page_len, b.first_page_offset, 0.3)
    o2, l2 = oracle.attention(q, b.k_pool[..., :D].contiguous(), b.v_pool[..., :D].contiguous(), b.indices,
                              b.indptr, b.last_page_len, b.first_page_offset, 0.3)
    fin = np.isfinite(l2)
    assert np.array_equal(np.isfinite(l1), fin)
    assert np.abs(o1 - o2).max() < 1e-12 and np.abs(l1[fin] - l2[fin]).max() < 1e-12


def test_concatenated_rows_equal_sdpa():
    b, q, qe, ke = _case(seed=3, dtype=torch.bfloat16)
    D = q.shape[2]
    scale = 1 / math.sqrt(D + ke.shape[3])
    o, l = oracle.attention_extra(q, qe, b.k_pool, ke, b.v_pool, D, b.indices, b.indptr, b.last_page_len,
                                  b.first_page_offset, scale)
    P, ps, Hkv, _ = b.k_pool.shape
    G = q.shape[1] // Hkv
    for r in range(q.shape[0]):
        n = b.seq_lens[r]
        rows = oracle.resolve_rows(b.indices, b.indptr, b.first_page_offset, ps, r, n)
        for kvh in range(Hkv):
            kc = torch.cat([b.k_pool.reshape(P * ps, Hkv, -1)[rows, kvh, :D],
                            ke.reshape(P * ps, Hkv, -1)[rows, kvh]], dim=1).double()
            v = b.v_pool.reshape(P * ps, Hkv, -1)[rows, kvh, :D].double()
            qc = torch.cat([q[r, kvh * G:(kvh + 1) * G], qe[r, kvh * G:(kvh + 1) * G]], dim=1).double()
            ref = torch.nn.functional.scaled_dot_product_attention(qc[None], kc[None], v[None], scale=scale)[0]
            lref = torch.logsumexp(scale * qc @ kc.T, dim=1) / math.log(2.0)
            assert float((torch.as_tensor(o[r, kvh * G:(kvh + 1) * G]) - ref).abs().max()) < 1e-12
            assert float((torch.as_tensor(l[r, kvh * G:(kvh + 1) * G]) - lref).abs().max()) < 1e-12


def test_closed_forms():
    b, q, qe, ke = _case(seed=5, seq=(1, 9, 4), fpo=(2, 0, 1))
    D = q.shape[2]
    o, l = oracle.attention_extra(q, qe, b.k_pool, ke, b.v_pool, D, b.indices, b.indptr, b.last_page_len,
                                  b.first_page_offset, 0.5)
    # request 0 sees one token: out = its V row, lse2 = its score in log2 units
    ps, Hkv = b.page_size, b.num_kv_heads
    row = oracle.resolve_rows(b.indices, b.indptr, b.first_page_offset, ps, 0, 1)[0]
    G = q.shape[1] // Hkv
    for h in range(q.shape[1]):
        kvh = h // G
        k = b.k_pool.reshape(-1, Hkv, b.k_pool.shape[3])[row, kvh, :D].double()
        kx = ke.reshape(-1, Hkv, ke.shape[3])[row, kvh].double()
        v = b.v_pool.reshape(-1, Hkv, b.v_pool.shape[3])[row, kvh, :D].double()
        s = 0.5 * (q[0, h].double() @ k + qe[0, h].double() @ kx)
        assert np.abs(o[0, h] - v.numpy()).max() == 0.0
        assert abs(l[0, h] - float(s) / math.log(2.0)) < 1e-12
    # an extra term that dominates one token of request 1 puts (almost) all the weight on it
    rows = oracle.resolve_rows(b.indices, b.indptr, b.first_page_offset, ps, 1, 9)
    ke2 = ke.clone().float()
    qe2 = qe.clone()
    qe2[1] = 0
    qe2[1, :, 0] = 1.0
    ke2.reshape(-1, Hkv, ke.shape[3])[rows[4], :, 0] = 1000.0
    o2, _ = oracle.attention_extra(q, qe2, b.k_pool, ke2.half(), b.v_pool, D, b.indices, b.indptr,
                                   b.last_page_len, b.first_page_offset, 0.5)
    for h in range(q.shape[1]):
        v = b.v_pool.reshape(-1, Hkv, b.v_pool.shape[3])[rows[4], h // G, :D].double().numpy()
        assert np.abs(o2[1, h] - v).max() < 1e-9


@pytest.mark.parametrize("ppc", [1, 2, 3, 4])
def test_partials_merge_to_the_whole(ppc):
    b, q, qe, ke = _case(seed=7, seq=(29, 7, 0), fpo=(3, 1, 0))
    D = q.shape[2]
    pl = oracle.plan(b.indptr, b.num_kv_heads, 1, 1, ppc)
    pv, plse = oracle.partials_extra(q, qe, b.k_pool, ke, b.v_pool, D, b.indices, b.indptr, b.last_page_len,
                                     b.first_page_offset, 0.4, ppc, pl.request_indices, pl.kv_tile_indices)
    mo, ml = oracle.merge(pv, plse, pl.o_indptr)
    o, l = oracle.attention_extra(q, qe, b.k_pool, ke, b.v_pool, D, b.indices, b.indptr, b.last_page_len,
                                  b.first_page_offset, 0.4)
    fin = np.isfinite(l)
    assert np.array_equal(np.isfinite(ml), fin)
    assert np.abs(mo - o).max() < 1e-12 and np.abs(ml[fin] - l[fin]).max() < 1e-12


def test_dsa_shaped_inputs_against_sdpa():
    """The DSA-shaped workload (128 heads, latent 512 + rope 64, values = latent rows, token-exact rows):
    the oracle against SDPA on the concatenated rows, request by request."""
    x = W.dsa_sparse_decode(batch=2, kv_len=1024, topk=256, heads=16)
    b = x.batch
    o, l = oracle.attention_extra(b.q, x.q_extra, b.k_pool, x.k_extra_pool, b.v_pool, x.dim, b.indices, b.indptr,
                                  b.last_page_len, b.first_page_offset, b.scale)
    for r in range(b.batch):
        rows = b.indices[b.indptr[r]:b.indptr[r + 1]].long()
        kc = torch.cat([b.k_pool[rows, 0, 0, :x.dim], x.k_extra_pool[rows, 0, 0]], dim=1).double()
        v = b.v_pool[rows, 0, 0, :x.dim].double()
        qc = torch.cat([b.q[r], x.q_extra[r]], dim=1).double()
        ref = torch.nn.functional.scaled_dot_product_attention(qc[None], kc[None], v[None], scale=b.scale)[0]
        assert float((torch.as_tensor(o[r]) - ref).abs().max()) < 1e-12
        assert float((torch.as_tensor(l[r]) - torch.logsumexp(b.scale * qc @ kc.T, 1) / math.log(2.0)).abs().max()) < 1e-12
