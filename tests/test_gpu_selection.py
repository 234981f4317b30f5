"""GPU: block -> token expansion (pa_selection_from_blocks) bit-exact against the oracle, and decodes over
the expanded (token-exact) and block-granular page tables against the oracle's attention."""
import random

import pytest
import torch

import oracle
from paged_attention_decode_gb300 import pa_v2 as pa
from paged_attention_decode_gb300 import workloads as W
from parity_helpers import assert_close

pytestmark = pytest.mark.gpu


def _expand(ids, C, kv_len, stride, status=None):
    return pa.pa_selection_from_blocks(ids.to("cuda"), C, kv_len, stride, status=status)


@pytest.mark.parametrize("C,kv_len,topk,R", [(4, 10, 2, 2), (1, 50, 30, 3), (3, 7, 0, 4), (128, 32731, 16, 4),
                                             (128, 32768, 16, 2), (64, 1000, 15, 16), (16, 4096 + 5, 255, 3)])
def test_expansion_is_bit_exact(C, kv_len, topk, R):
    rng = random.Random(C * 7919 + kv_len)
    nb = -(-kv_len // C)
    ids = torch.tensor([rng.sample(range(nb - 1), topk) for _ in range(R)], dtype=torch.int32).reshape(R, topk)
    stride = kv_len + rng.randint(0, 300)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _expand(ids, C, kv_len, stride, status)
    ref, per = oracle.selection_rows_ref(ids, C, kv_len, stride)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert got.numel() == R * per
    assert torch.equal(got.cpu(), ref)


def test_expansion_reports_out_of_range_block_ids():
    C, kv_len = 8, 40                                     # nb = 5: scored blocks 0..3
    ids = torch.tensor([[1, 4], [0, -1], [3, 2]], dtype=torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _expand(ids, C, kv_len, 64, status).cpu()
    torch.cuda.synchronize()
    assert int(status.item()) & pa.DEVICE_BAD_BLOCK
    per = 2 * C + 8
    # the bad blocks' rows are -1; everything else is the oracle's
    ref, _ = oracle.selection_rows_ref(torch.tensor([[1, 0], [0, 0], [3, 2]], dtype=torch.int32), C, kv_len, 64)
    for r, bad_slot in ((0, 1), (1, 1), (2, None)):
        row = got[r * per:(r + 1) * per]
        for slot in range(2):
            seg = row[slot * C:(slot + 1) * C]
            if slot == bad_slot:
                assert torch.all(seg == -1)
            else:
                assert torch.equal(seg, ref[r * per + slot * C:r * per + (slot + 1) * C])
        assert torch.equal(row[2 * C:], ref[r * per + 2 * C:(r + 1) * per])


def _decode(plan, q, kp, vp, idx, ip, lp, fp, scale):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, l = pa.decode(plan, q, kp, vp, idx, ip, lp, fp, scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return o, l


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_token_exact_decode_over_expanded_rows(dtype):
    s = W.block_sparse_selection(dtype=dtype, kv_len=8191, cap=8448, topk=12)
    d = s.to("cuda")
    R, n_rep, D = s.q.shape
    rows = pa.pa_selection_from_blocks(d.block_ids, s.block_size, s.kv_len, s.cap)
    per = pa.pa_selection_rows_per_request(s.block_ids.shape[1], s.block_size, s.kv_len)
    ip, lp, fp = pa.pa_sparse_csr(R, per)
    dt = pa.KV_DTYPES[dtype]
    plan = pa.pa_v2_plan(ip, lp, fp, 1, n_rep, 1, D, dt, pa.pa_v2_default_target_ctas(n_rep, 1, D, 1, dt))
    o, l = _decode(plan, d.q, d.k_pool, d.v_pool, rows, ip.cuda(), lp.cuda(), fp.cuda(), s.scale)
    ref_rows, _ = oracle.selection_rows_ref(s.block_ids, s.block_size, s.kv_len, s.cap)
    ro, rl = oracle.attention(s.q, s.k_pool, s.v_pool, ref_rows, ip, lp, fp, s.scale)
    assert_close(o, l, ro, rl, "token-exact selection")


def test_block_granular_decode_matches_token_exact():
    """Pool-backed cache: the selected block ids as pages of block_size rows (final block last)."""
    s = W.block_sparse_selection(kv_len=8191, cap=8448, topk=12)
    R, n_rep, D = s.q.shape
    C = s.block_size
    bpr = s.cap // C
    pages, ip, lp, fp = oracle.selection_pages_ref(s.block_ids, C, s.kv_len, bpr)
    kp = s.k_pool.reshape(R * bpr, C, 1, D)
    vp = s.v_pool.reshape(R * bpr, C, 1, D)
    dt = pa.PA_F16
    plan = pa.pa_v2_plan(ip, lp, fp, C, n_rep, 1, D, dt, pa.pa_v2_default_target_ctas(n_rep, 1, D, C, dt))
    o, l = _decode(plan, s.q.cuda(), kp.cuda(), vp.cuda(), pages.cuda(), ip.cuda(), lp.cuda(), fp.cuda(), s.scale)
    ref_rows, per = oracle.selection_rows_ref(s.block_ids, C, s.kv_len, s.cap)
    ip1, lp1, fp1 = oracle.sparse_csr_ref(R, per)
    ro, rl = oracle.attention(s.q, s.k_pool, s.v_pool, ref_rows, ip1, lp1, fp1, s.scale)
    assert_close(o, l, ro, rl, "block-granular selection")
