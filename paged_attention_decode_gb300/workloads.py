"""Seeded synthetic inputs for paged-attention decode.

This module only builds inputs: a CSR page table over a paged KV pool, the
pools themselves and the query.  It holds none of the attention arithmetic
and imports neither the CUDA binding nor the oracle, so the GPU path and the
oracle can both be fed from it.

Layouts (issue #898, Task 1 and design piece 1; PR #984, What changed 1):

- ``k_pool``/``v_pool``: ``[num_pages, page_size, num_kv_heads, head_dim]``,
  one contiguous buffer per side.
- ``indices`` (int32, flat physical page ids), ``indptr`` (int32, ``[B+1]``),
  ``last_page_len`` (int32, ``[B]``, valid entries of the final page, equal to
  ``page_size`` when that page is exactly full) and ``first_page_offset``
  (int32, ``[B]``, the entry of the first page where a sliding window starts).
- ``q``: ``[B, Hq, head_dim]`` float32.

All random values are N(0, 1) from a CPU ``torch.Generator`` seeded per
workload, cast to the pool dtype; consumers read the cast values.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Sequence

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
DTYPE_NAMES = {v: k for k, v in DTYPES.items()}


@dataclass
class PagedBatch:
    """One decode step's inputs (all tensors on the CPU)."""

    name: str
    q: torch.Tensor
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    indices: torch.Tensor
    indptr: torch.Tensor
    last_page_len: torch.Tensor
    first_page_offset: torch.Tensor
    seq_lens: list[int]
    page_size: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    scale: float
    ppc_override: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return len(self.seq_lens)

    @property
    def num_pages(self) -> int:
        return self.k_pool.shape[0]

    @property
    def dtype(self) -> torch.dtype:
        return self.k_pool.dtype

    def kv_bytes(self) -> int:
        """Bytes of K and V the step must read: every visible token, every KV head, both sides."""
        return sum(self.seq_lens) * self.num_kv_heads * self.head_dim * 2 * self.k_pool.element_size()

    def to(self, device) -> "PagedBatch":
        moved = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in self.__dict__.items()}
        return PagedBatch(**moved)


def page_geometry(seq_len: int, first_page_offset: int, page_size: int) -> tuple[int, int]:
    """(pages, last_page_len) of a request whose window starts at entry ``first_page_offset``.

    A request with no visible token owns no page and has last_page_len 0.
    """
    if seq_len == 0:
        return 0, 0
    end = first_page_offset + seq_len          # entries used, counted from the first page's entry 0
    pages = -(-end // page_size)
    return pages, end - (pages - 1) * page_size


def _randn(gen: torch.Generator, shape, dtype: torch.dtype) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(dtype)


def make_batch(name: str, seq_lens: Sequence[int], first_page_offsets: Sequence[int], page_size: int,
               num_qo_heads: int, num_kv_heads: int, head_dim: int, dtype: torch.dtype, seed: int,
               slack: float = 2.0, num_pages: int | None = None, order: str = "shuffled",
               scale: float | None = None, ppc_override: int = 0) -> PagedBatch:
    """A batch whose requests own disjoint physical pages drawn from a pool with slack.

    ``order``: "shuffled" (a random permutation of pool pages), "reversed"
    (pages handed out from the top of the pool downwards) or "identity"
    (contiguous ascending pages).
    """
    gen = torch.Generator().manual_seed(seed)
    B = len(seq_lens)
    geo = [page_geometry(s, f, page_size) for s, f in zip(seq_lens, first_page_offsets)]
    total = sum(p for p, _ in geo)
    P = num_pages if num_pages is not None else max(1, int(math.ceil(total * slack)))
    assert P >= total, "pool too small for the batch"
    if order == "shuffled":
        ids = torch.randperm(P, generator=gen)[:total]
    elif order == "reversed":
        ids = torch.arange(P - 1, P - 1 - total, -1)
    elif order == "identity":
        ids = torch.arange(total)
    else:
        raise ValueError(order)
    indptr = [0]
    for p, _ in geo:
        indptr.append(indptr[-1] + p)
    q = torch.randn(B, num_qo_heads, head_dim, generator=gen, dtype=torch.float32)
    k_pool = _randn(gen, (P, page_size, num_kv_heads, head_dim), dtype)
    v_pool = _randn(gen, (P, page_size, num_kv_heads, head_dim), dtype)
    return PagedBatch(
        name=name, q=q, k_pool=k_pool, v_pool=v_pool,
        indices=ids.to(torch.int32),
        indptr=torch.tensor(indptr, dtype=torch.int32),
        last_page_len=torch.tensor([l for _, l in geo], dtype=torch.int32),
        first_page_offset=torch.tensor([f if s > 0 else 0 for s, f in zip(seq_lens, first_page_offsets)],
                                       dtype=torch.int32),
        seq_lens=list(seq_lens), page_size=page_size, num_qo_heads=num_qo_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim,
        scale=scale if scale is not None else 1.0 / math.sqrt(head_dim),
        ppc_override=ppc_override)


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------

def tiny_csr(seed: int = 1000) -> PagedBatch:
    """B=2, Hq=4, Hkv=2, D=64, page_size=4, seq_lens {13, 7}, first_page_offset {0, 2},
    a 16-page fp32 pool with shuffled page ids, chunks fixed at 2 pages then merged."""
    return make_batch("tiny_csr", [13, 7], [0, 2], page_size=4, num_qo_heads=4, num_kv_heads=2,
                      head_dim=64, dtype=torch.float32, seed=seed, num_pages=16, ppc_override=2)


def llama3_8b_32k(seed: int = 1001, context: int = 32768) -> PagedBatch:
    """Llama-3-8B-shaped single-sequence decode: B=1, Hq=32, Hkv=8, D=128, fp16 pools,
    page_size=16, 32768 tokens on a random permutation of a pool with 2x slack."""
    return make_batch("llama3_8b_32k", [context], [0], page_size=16, num_qo_heads=32, num_kv_heads=8,
                      head_dim=128, dtype=torch.float16, seed=seed, slack=2.0)


def sliding_window_batch(seed: int = 1002) -> PagedBatch:
    """B=4, Hq=32, Hkv=8, D=128, bf16, page_size=16.  Requests 0-1 are 4096-token windows
    starting mid-page (first_page_offset uniform in [1, 15], retired pages not in the table);
    requests 2-3 have seq_len uniform in [1024, 16384] starting at entry 0."""
    gen = torch.Generator().manual_seed(seed)
    fpo = [int(torch.randint(1, 16, (1,), generator=gen)) for _ in range(2)] + [0, 0]
    lens = [4096, 4096] + [int(torch.randint(1024, 16385, (1,), generator=gen)) for _ in range(2)]
    return make_batch("sliding_window_batch", lens, fpo, page_size=16, num_qo_heads=32, num_kv_heads=8,
                      head_dim=128, dtype=torch.bfloat16, seed=seed + 7, slack=2.0)


def sparse_token_exact(seed: int = 1003, batch: int = 2, heads: int = 8, cap: int = 131072,
                       head_dim: int = 128, n_rep: int = 4, selected: int = 2048) -> PagedBatch:
    """Token-exact sparse decode at page_size=1 (sparse-paged-decode.md, issue #904).

    A dense fp16 cache [batch, heads, cap, head_dim] per side is viewed, without a copy, as the
    pool [batch*heads*cap, 1, 1, head_dim].  KV heads fold into requests (r = b*heads + h), each
    with n_rep query heads; a request's page list is its ``selected`` sorted unique positions,
    drawn uniformly without replacement, offset by the head stride ``cap``."""
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn(batch, heads * n_rep, head_dim, generator=gen, dtype=torch.float32)
    k = torch.empty(batch, heads, cap, head_dim, dtype=torch.float16)
    v = torch.empty(batch, heads, cap, head_dim, dtype=torch.float16)
    for b in range(batch):
        for h in range(heads):
            k[b, h] = torch.randn(cap, head_dim, generator=gen).half()
            v[b, h] = torch.randn(cap, head_dim, generator=gen).half()
    positions = []
    for r in range(batch * heads):
        pos = torch.randperm(cap, generator=gen)[:selected].sort().values
        positions.append(pos)
    indices = torch.cat([r * cap + p for r, p in enumerate(positions)]).to(torch.int32)
    R = batch * heads
    return PagedBatch(
        name="sparse_token_exact", q=q.reshape(R, n_rep, head_dim),
        k_pool=k.reshape(batch * heads * cap, 1, 1, head_dim),
        v_pool=v.reshape(batch * heads * cap, 1, 1, head_dim),
        indices=indices,
        indptr=torch.arange(0, (R + 1) * selected, selected, dtype=torch.int32),
        last_page_len=torch.ones(R, dtype=torch.int32),
        first_page_offset=torch.zeros(R, dtype=torch.int32),
        seq_lens=[selected] * R, page_size=1, num_qo_heads=n_rep, num_kv_heads=1,
        head_dim=head_dim, scale=1.0 / math.sqrt(head_dim),
        meta={"positions": positions, "cap": cap, "dense_shape": (batch, heads, cap, head_dim)})


@dataclass
class CascadeBatch:
    """M requests sharing a whole-page prefix: the flat batch plus both cascade levels' tables."""

    flat: PagedBatch
    prefix_indices: torch.Tensor        # [shared_pages] int32, full pages
    suffix_indices: torch.Tensor        # flat page ids of the private suffixes
    suffix_indptr: torch.Tensor         # [M+1]
    suffix_last_page_len: torch.Tensor  # [M]
    suffix_lens: list[int]


def cascade_shared_prefix(seed: int = 1004, members: int = 4, prefix_tokens: int = 8192,
                          suffix_range: tuple[int, int] = (256, 2048), num_qo_heads: int = 32,
                          num_kv_heads: int = 8, head_dim: int = 128, page_size: int = 16,
                          dtype: torch.dtype = torch.float16) -> CascadeBatch:
    """Cascade workload (cascade-attention.md, issue #903): M members share a prefix of
    identical page ids; private suffixes of uniform length on private pages."""
    assert prefix_tokens % page_size == 0, "the shared span is whole pages"
    gen = torch.Generator().manual_seed(seed)
    suffix_lens = [int(torch.randint(suffix_range[0], suffix_range[1] + 1, (1,), generator=gen))
                   for _ in range(members)]
    npre = prefix_tokens // page_size
    sgeo = [page_geometry(s, 0, page_size) for s in suffix_lens]
    total = npre + sum(p for p, _ in sgeo)
    P = 2 * total
    ids = torch.randperm(P, generator=gen)[:total].to(torch.int32)
    prefix = ids[:npre]
    suffix = ids[npre:]
    sindptr = [0]
    for p, _ in sgeo:
        sindptr.append(sindptr[-1] + p)
    flat_indices, flat_indptr = [], [0]
    for m in range(members):
        own = torch.cat([prefix, suffix[sindptr[m]:sindptr[m + 1]]])
        flat_indices.append(own)
        flat_indptr.append(flat_indptr[-1] + len(own))
    q = torch.randn(members, num_qo_heads, head_dim, generator=gen, dtype=torch.float32)
    k_pool = _randn(gen, (P, page_size, num_kv_heads, head_dim), dtype)
    v_pool = _randn(gen, (P, page_size, num_kv_heads, head_dim), dtype)
    lpl = torch.tensor([l for _, l in sgeo], dtype=torch.int32)
    flat = PagedBatch(
        name="cascade_shared_prefix", q=q, k_pool=k_pool, v_pool=v_pool,
        indices=torch.cat(flat_indices), indptr=torch.tensor(flat_indptr, dtype=torch.int32),
        last_page_len=lpl.clone(), first_page_offset=torch.zeros(members, dtype=torch.int32),
        seq_lens=[prefix_tokens + s for s in suffix_lens], page_size=page_size,
        num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
        scale=1.0 / math.sqrt(head_dim), meta={"prefix_tokens": prefix_tokens})
    return CascadeBatch(flat=flat, prefix_indices=prefix, suffix_indices=suffix,
                        suffix_indptr=torch.tensor(sindptr, dtype=torch.int32),
                        suffix_last_page_len=lpl, suffix_lens=suffix_lens)


def cascade_mixed_batch(seed: int = 1005, prefix_tokens: int = 2048, num_qo_heads: int = 16, num_kv_heads: int = 4,
                        head_dim: int = 128, page_size: int = 16, dtype: torch.dtype = torch.float16) -> PagedBatch:
    """A flat batch in which some requests share a whole-page prefix and others do not.

    Requests 0, 2 and 5 share the first prefix_tokens / page_size page ids and then have private
    suffixes; request 3 holds the same pages but its window starts mid-page (first_page_offset 5);
    requests 1 and 4 share nothing."""
    gen = torch.Generator().manual_seed(seed)
    npre = prefix_tokens // page_size
    kinds = ["member", "other", "member", "midpage", "other", "member"]
    lens = [int(torch.randint(100, 1500, (1,), generator=gen)) for _ in kinds]
    P = 4 * (npre + sum(-(-(L + 16) // page_size) for L in lens) + 8)
    ids = torch.randperm(P, generator=gen).to(torch.int32)
    prefix = ids[:npre]
    nxt = npre
    tables, fpos, seq = [], [], []
    for kind, L in zip(kinds, lens):
        if kind == "other":
            pg, lpl = page_geometry(L, 0, page_size)
            tables.append(ids[nxt:nxt + pg])
            nxt += pg
            fpos.append(0)
            seq.append(L)
        else:
            f = 5 if kind == "midpage" else 0
            total = prefix_tokens - f + L
            pg, lpl = page_geometry(total, f, page_size)
            own = pg - npre
            tables.append(torch.cat([prefix, ids[nxt:nxt + own]]))
            nxt += own
            fpos.append(f)
            seq.append(total)
    indptr = [0]
    for t in tables:
        indptr.append(indptr[-1] + len(t))
    geo = [page_geometry(L, f, page_size) for L, f in zip(seq, fpos)]
    q = torch.randn(len(kinds), num_qo_heads, head_dim, generator=gen, dtype=torch.float32)
    k_pool = _randn(gen, (P, page_size, num_kv_heads, head_dim), dtype)
    v_pool = _randn(gen, (P, page_size, num_kv_heads, head_dim), dtype)
    return PagedBatch(
        name="cascade_mixed_batch", q=q, k_pool=k_pool, v_pool=v_pool, indices=torch.cat(tables),
        indptr=torch.tensor(indptr, dtype=torch.int32),
        last_page_len=torch.tensor([l for _, l in geo], dtype=torch.int32),
        first_page_offset=torch.tensor(fpos, dtype=torch.int32), seq_lens=seq, page_size=page_size,
        num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads, head_dim=head_dim, scale=1.0 / math.sqrt(head_dim),
        meta={"members": [0, 2, 5], "shared_pages": npre})


def scatter_dense(name: str, dense_k: Sequence[torch.Tensor], dense_v: Sequence[torch.Tensor],
                  first_page_offsets: Sequence[int], page_size: int, num_qo_heads: int,
                  seed: int, slack: float = 2.0, order: str = "shuffled",
                  dtype: torch.dtype = torch.float32, fill: float = float("nan")) -> PagedBatch:
    """Write given dense per-request sequences ``[L_r, Hkv, D]`` into a paged pool.

    Request r's token i is written to page entry (first_page_offset[r] + i) mod page_size of its
    ((first_page_offset[r] + i) div page_size)-th page; every other pool entry holds ``fill``,
    so any read outside the sequences shows up.  This is the construction the page-resolution
    rule inverts, used to pin it from the other side.
    """
    gen = torch.Generator().manual_seed(seed)
    lens = [int(k.shape[0]) for k in dense_k]
    Hkv, D = dense_k[0].shape[1], dense_k[0].shape[2]
    geo = [page_geometry(L, f, page_size) for L, f in zip(lens, first_page_offsets)]
    total = sum(p for p, _ in geo)
    P = max(1, int(math.ceil(total * slack)))
    if order == "shuffled":
        ids = torch.randperm(P, generator=gen)[:total]
    elif order == "reversed":
        ids = torch.arange(P - 1, P - 1 - total, -1)
    else:
        ids = torch.arange(total)
    k_pool = torch.full((P, page_size, Hkv, D), fill, dtype=dtype)
    v_pool = torch.full((P, page_size, Hkv, D), fill, dtype=dtype)
    indptr = [0]
    for r, (L, f) in enumerate(zip(lens, first_page_offsets)):
        base = indptr[-1]
        for i in range(L):
            page = int(ids[base + (f + i) // page_size])
            k_pool[page, (f + i) % page_size] = dense_k[r][i].to(dtype)
            v_pool[page, (f + i) % page_size] = dense_v[r][i].to(dtype)
        indptr.append(base + geo[r][0])
    q = torch.randn(len(lens), num_qo_heads, D, generator=gen, dtype=torch.float32)
    return PagedBatch(
        name=name, q=q, k_pool=k_pool, v_pool=v_pool, indices=ids.to(torch.int32),
        indptr=torch.tensor(indptr, dtype=torch.int32),
        last_page_len=torch.tensor([l for _, l in geo], dtype=torch.int32),
        first_page_offset=torch.tensor([f if L > 0 else 0 for L, f in zip(lens, first_page_offsets)],
                                       dtype=torch.int32),
        seq_lens=lens, page_size=page_size, num_qo_heads=num_qo_heads, num_kv_heads=Hkv,
        head_dim=D, scale=1.0 / math.sqrt(D))


@dataclass
class BlockSelection:
    """A block-sparse decode input: a dense cache [B, H, cap, D] per side viewed as the page_size-1 pool
    [B*H*cap, 1, 1, D], requests r = b*H + h (n_rep query heads each), and each request's selected block
    ids -- distinct, unordered (as an argpartition returns them), drawn from the scored blocks
    0 .. nb-2 of the live window kv_len, nb = ceil(kv_len / block_size).  Expanding the ids into rows is
    the method's work and is not done here."""

    q: torch.Tensor            # [R, n_rep, D] f32
    k_pool: torch.Tensor       # [B*H*cap, 1, 1, D]
    v_pool: torch.Tensor
    block_ids: torch.Tensor    # [R, topk] int32
    block_size: int
    kv_len: int
    cap: int
    scale: float
    name: str = "block_sparse_selection"

    @property
    def num_requests(self) -> int:
        return self.q.shape[0]

    def to(self, device) -> "BlockSelection":
        return BlockSelection(self.q.to(device), self.k_pool.to(device), self.v_pool.to(device),
                              self.block_ids.to(device), self.block_size, self.kv_len, self.cap, self.scale, self.name)


def block_sparse_selection(seed: int = 1006, batch: int = 1, kv_heads: int = 4, n_rep: int = 16, head_dim: int = 128,
                           kv_len: int = 32731, cap: int = 33024, block_size: int = 128, topk: int = 16,
                           dtype: torch.dtype = torch.float16) -> BlockSelection:
    """MiniMax-M3-shaped block-sparse decode (sparse-paged-decode.md: 64 query heads over 4 KV heads,
    head_dim 128, block_size 128, topk_blocks 16).  kv_len leaves a partial final block (91 rows at the
    defaults); cap, the reserved capacity, exceeds kv_len (33024 = 258 blocks, so the same allocation also
    serves as a pool of 128-row pages)."""
    gen = torch.Generator().manual_seed(seed)
    R = batch * kv_heads
    nb = -(-kv_len // block_size)
    q = torch.randn(R, n_rep, head_dim, generator=gen, dtype=torch.float32)
    k = torch.randn(R * cap, 1, 1, head_dim, generator=gen).to(dtype)
    v = torch.randn(R * cap, 1, 1, head_dim, generator=gen).to(dtype)
    ids = torch.stack([torch.randperm(nb - 1, generator=gen)[:topk] for _ in range(R)]).to(torch.int32)
    return BlockSelection(q, k, v, ids, block_size, kv_len, cap, 1.0 / math.sqrt(head_dim))


@dataclass
class ExtraStreamBatch:
    """Decode input for the second-K-stream kernel: a PagedBatch whose k_pool rows are RowStride wide (the
    first `dim` elements are the key; v_pool may be the same tensor), plus q_extra and k_extra_pool."""

    batch: PagedBatch
    q_extra: torch.Tensor       # [B, Hq, extra]
    k_extra_pool: torch.Tensor  # [P, page_size, Hkv, extra]
    dim: int
    shared_v: bool

    def to(self, device) -> "ExtraStreamBatch":
        b = self.batch.to(device)
        if self.shared_v:
            b.v_pool = b.k_pool
        return ExtraStreamBatch(b, self.q_extra.to(device), self.k_extra_pool.to(device), self.dim, self.shared_v)


def dsa_sparse_decode(seed: int = 1007, batch: int = 4, heads: int = 128, kv_lora_rank: int = 512,
                      index_head_dim: int = 128, rope_dim: int = 64, kv_len: int = 8192, topk: int = 2048,
                      dtype: torch.dtype = torch.bfloat16) -> ExtraStreamBatch:
    """DSA-shaped token-exact sparse decode (sparse-paged-decode.md, the DSA paragraphs): per sequence a K
    allocation [cap, kv_lora_rank + index_head_dim] (concat(kv_latent, indexer_key)) and a k_pe allocation
    [cap, rope_dim], one KV head (MLA), `heads` query heads with q_latent [.., kv_lora_rank] and q_pe
    [.., rope_dim]; the values are the latent rows (v_pool is k_pool).  Each request selects `topk` sorted
    unique positions of its live window (an indexer's top-k), offset by the row stride cap between
    sequences.  Scale 1/sqrt(128 + rope_dim): DeepSeek's qk head dim (nope 128 + rope)."""
    gen = torch.Generator().manual_seed(seed)
    cap = kv_len + 256
    width = kv_lora_rank + index_head_dim
    k = torch.randn(batch * cap, 1, 1, width, generator=gen).to(dtype)
    kpe = torch.randn(batch * cap, 1, 1, rope_dim, generator=gen).to(dtype)
    q = torch.randn(batch, heads, kv_lora_rank, generator=gen, dtype=torch.float32)
    qe = torch.randn(batch, heads, rope_dim, generator=gen, dtype=torch.float32)
    sel = [torch.randperm(kv_len, generator=gen)[:topk].sort().values + r * cap for r in range(batch)]
    pb = PagedBatch(
        name="dsa_sparse_decode", q=q, k_pool=k, v_pool=k, indices=torch.cat(sel).to(torch.int32),
        indptr=torch.arange(0, (batch + 1) * topk, topk, dtype=torch.int32),
        last_page_len=torch.ones(batch, dtype=torch.int32), first_page_offset=torch.zeros(batch, dtype=torch.int32),
        seq_lens=[topk] * batch, page_size=1, num_qo_heads=heads, num_kv_heads=1, head_dim=kv_lora_rank,
        scale=1.0 / math.sqrt(128 + rope_dim), meta={"cap": cap, "kv_len": kv_len})
    return ExtraStreamBatch(pb, qe, kpe, kv_lora_rank, True)


WORKLOADS = {
    "tiny_csr": tiny_csr,
    "llama3_8b_32k": llama3_8b_32k,
    "sliding_window_batch": sliding_window_batch,
    "sparse_token_exact": sparse_token_exact,
    "cascade_shared_prefix": cascade_shared_prefix,
}
