"""GPU: a decode launched right after a kernel that rewrites its page table reads the new table.

The partial kernel runs as a programmatic dependent of the kernel before it, and a one-request plan's CTAs
read their first page ids speculatively before waiting for that kernel (to warm L2; issue #898 design
piece 2 is the kernel this touches).  Those reads may see the table half rewritten; they must only ever
choose prefetch addresses.  Here pa_selection_from_blocks -- itself a programmatic launch that releases its
dependents at entry -- overwrites the page-id buffer with selection A or B in turn, each time right before
a one-request decode over it, so the buffer always holds the other selection's valid ids while the decode
starts.  Every step must match the oracle's attention over the selection written just before it.
"""
import random

import pytest
import torch

import oracle
from paged_attention_decode_gb300 import pa_v2 as pa
from parity_helpers import assert_close

pytestmark = pytest.mark.gpu

STEPS = 12


def _case(page_size):
    """(pool, q, block size, kv_len, two selections as [1, topk] int32) for one request."""
    g = torch.Generator().manual_seed(4100 + page_size)
    if page_size == 16:
        # block size 1 over kv_len = P positions: the selection's rows are page ids of a 16-row-page pool
        P, Hkv, D, Hq, C, kv_len, topk = 1024, 8, 128, 32, 1, 1024, 255
    else:
        # token rows of a page_size-1 pool (the token-exact layout)
        P, Hkv, D, Hq, C, kv_len, topk = 8192, 8, 128, 32, 64, 8192, 24
    k = torch.randn(P, page_size, Hkv, D, generator=g).to(torch.float16)
    v = torch.randn(P, page_size, Hkv, D, generator=g).to(torch.float16)
    q = torch.randn(1, Hq, D, generator=g)
    nb = -(-kv_len // C)
    rng = random.Random(page_size)
    sels = [torch.tensor([rng.sample(range(nb - 1), topk)], dtype=torch.int32) for _ in range(2)]
    return k, v, q, C, kv_len, sels


@pytest.mark.parametrize("page_size", [16, 1])
@pytest.mark.parametrize("graph", [False, True])
def test_decode_after_a_kernel_that_rewrites_its_page_table(page_size, graph):
    k, v, q, C, kv_len, sels = _case(page_size)
    Hq, D = q.shape[1], q.shape[2]
    Hkv = k.shape[2]
    per = pa.pa_selection_rows_per_request(sels[0].shape[1], C, kv_len)
    last = page_size if page_size > 1 else 1
    ip, lp, fp = torch.tensor([0, per], dtype=torch.int32), torch.tensor([last], dtype=torch.int32), \
        torch.zeros(1, dtype=torch.int32)
    dt = pa.PA_F16
    plan = pa.pa_v2_plan(ip, lp, fp, page_size, Hq, Hkv, D, dt,
                         pa.pa_v2_default_target_ctas(Hq, Hkv, D, page_size, dt))
    assert plan.batch == 1 and plan.num_chunks > 1
    refs = []
    for sel in sels:
        rows, n = oracle.selection_rows_ref(sel, C, kv_len, kv_len)
        assert n == per
        refs.append(oracle.attention(q, k, v, rows, ip, lp, fp, 0.088))
    dev = torch.device("cuda")
    kd, vd, qd = k.to(dev), v.to(dev), q.to(dev)
    ipd, lpd, fpd = ip.to(dev), lp.to(dev), fp.to(dev)
    idsd = [s.to(dev) for s in sels]
    s = plan.struct
    ws = (torch.empty(s.num_chunks, Hq, D, device=dev), torch.empty(s.num_chunks, Hq, device=dev))
    idx = torch.empty(per, dtype=torch.int32, device=dev)
    outs = torch.empty(STEPS, 1, Hq, D, device=dev)
    lses = torch.empty(STEPS, 1, Hq, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream()

    def steps():
        for t in range(STEPS):
            pa.pa_selection_from_blocks(idsd[t % 2], C, kv_len, kv_len, indices=idx, status=status, stream=stream)
            pa.decode(plan, qd, kd, vd, idx, ipd, lpd, fpd, 0.088, out=outs[t], lse2=lses[t], workspace=ws,
                      status=status, stream=stream)

    with torch.cuda.stream(stream):
        pa.pa_selection_from_blocks(idsd[1], C, kv_len, kv_len, indices=idx, status=status, stream=stream)
        if graph:
            steps()                                   # warm-up, then capture the same launches
            stream.synchronize()
            outs.zero_()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                steps()
            for _ in range(2):
                g.replay()
        else:
            steps()
    stream.synchronize()
    assert int(status.item()) == 0
    for t in range(STEPS):
        ro, rl = refs[t % 2]
        assert_close(outs[t].cpu(), lses[t].cpu(), ro, rl, f"step {t} (selection {'AB'[t % 2]})")
    # the two selections give different results, so a step that read the other one would have failed
    assert (outs[0] - outs[1]).abs().max().item() > 1e-2
