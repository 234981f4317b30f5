"""Host side of the block-sparse selection entry points (no GPU): the row count and the CSR structure
against the oracle, and argument rejection."""
import random

import pytest
import torch

import oracle
from paged_attention_decode_gb300 import pa_v2 as pa


def test_rows_per_request_matches_the_oracle():
    rng = random.Random(21)
    for _ in range(500):
        C = rng.choice([1, 2, 3, 16, 64, 128])
        kv_len = rng.randint(1, 5000)
        nb = -(-kv_len // C)
        topk = rng.randint(0, nb - 1)
        ids = torch.tensor([rng.sample(range(nb - 1), topk)], dtype=torch.int32).reshape(1, topk)
        _, per = oracle.selection_rows_ref(ids, C, kv_len, kv_len)
        assert pa.pa_selection_rows_per_request(topk, C, kv_len) == per


@pytest.mark.parametrize("args", [(3, 4, 10), (0, 0, 5), (-1, 4, 10), (0, 4, 0), (1, 5, 5)])
def test_rows_per_request_rejects_invalid_arguments(args):
    with pytest.raises(pa.PaError):
        pa.pa_selection_rows_per_request(*args)


@pytest.mark.parametrize("R,per", [(0, 0), (1, 1), (3, 7), (16, 2048), (5, 0)])
def test_sparse_csr_matches_the_oracle(R, per):
    got = pa.pa_sparse_csr(R, per)
    ref = oracle.sparse_csr_ref(R, per)
    for g, r in zip(got, ref):
        assert g.tolist() == r.tolist()


def test_sparse_csr_rejects_overflow_and_negatives():
    for R, per in ((-1, 3), (2, -1), (3, 1 << 30)):
        with pytest.raises(pa.PaError):
            pa.pa_sparse_csr(R, per)


def test_device_status_bit_for_bad_blocks_maps_to_eoob():
    assert pa.pa_status_from_device(pa.DEVICE_BAD_BLOCK) == pa.PA_EOOB



@pytest.mark.parametrize("G", [1, 4, 16, 20, 128])
def test_heads_per_cta_rule_for_the_second_k_stream(G):
    for dt in (pa.PA_F16, pa.PA_BF16):
        assert pa.pa_v2_q_heads_per_cta(G, 512, dt) == min(G, 32)
    assert pa.pa_v2_q_heads_per_cta(G, 512, pa.PA_F32) == 0
    assert pa.pa_v2_q_heads_per_cta(G, 256, pa.PA_F16) == 0
