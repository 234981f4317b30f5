"""Plain f64 CPU oracle for fused paged-attention decode v2.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s cpu_baseline / ``--impl reference`` legs import this package.
The product path (``paged_attention_decode_gb300``) never imports it, and the
two share no code: the arithmetic lives in ``pa_oracle.c`` (plain C, double
precision, see its header for the passage each function follows) and this
module only marshals arrays into it.

Cascade composition (``cascade_ref``) follows cascade-attention.md (issue
#903): level 0 attends the shared span once with the members' query heads
stacked ``h0 = kv * (M * G) + m * G + g``, level 1 attends each member's
private suffix, and one merge pairs each member's two states.
``cascade_detect_ref`` is that page's detection rule written as plain loops.

Block-sparse selections (sparse-paged-decode.md, issue #904: the paragraphs on
``selection_from_blocks`` and on the final block): ``selection_rows_ref``
expands the selected block ids of each request into the token rows a
token-exact (page_size 1) page table lists, and ``selection_pages_ref`` gives
the block-granular (page_size = block size) page list of a pool-backed cache.
Both are plain loops over integers.

Second K stream (sparse-paged-decode.md, the DSA paragraphs, third way out):
``attention_extra`` scores token t as scale * (q . k[row_t][:dim] + q_extra .
k_extra[row_t][:extra_dim]) and averages v[row_t][:dim]; rows resolve through
the same page table as every other decode.  It gathers the rows with the
pinned page resolution and uses f64 matrix products (a library primitive) for
the two dot products and the weighted sum.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_pa.so")

DTYPE_CODES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}

# geometry validation codes, mirroring the enum in pa_oracle.c
GEOM_OK = 0
GEOM_BAD_ARGS = 1
GEOM_INDPTR0 = 2
GEOM_INDPTR_ORDER = 3
GEOM_LAST_PAGE_LEN = 4
GEOM_FIRST_OFFSET = 5
GEOM_SINGLE_PAGE = 6
GEOM_EMPTY_REQUEST = 7
GEOM_PAGE_ID = 8
GEOM_IDENTITY = 9

MAX_CHUNKS = 65535


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into liboracle_pa.so next to it (gcc, OpenMP if available)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
            "-D_GNU_SOURCE", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        P, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        L.ora_decode_element.argtypes = [P, i32, i64]
        L.ora_decode_element.restype = f64
        L.ora_num_threads.restype = i32
        L.ora_seq_len.argtypes = [P, P, P, i32, i32]
        L.ora_seq_len.restype = i64
        L.ora_validate_geometry.argtypes = [P, P, P, i32, i32, P, i64, P]
        L.ora_validate_geometry.restype = i32
        L.ora_resolve_row.argtypes = [P, P, P, i32, i32, i64]
        L.ora_resolve_row.restype = i64
        L.ora_attention.argtypes = [P, P, P, i32, P, P, P, P, i32, i32, i32, i32, i32, f64, P, P]
        L.ora_attention.restype = None
        L.ora_partials.argtypes = [P, P, P, i32, P, P, P, P, i32, i32, i32, i32, i32, P, P, i64, f64, P, P]
        L.ora_partials.restype = None
        L.ora_merge.argtypes = [P, P, P, i32, i32, i32, P, P]
        L.ora_merge.restype = None
        L.ora_plan.argtypes = [P, i32, i32, i32, i64, i32, i64, P, P, P, P, P, P, i64, P]
        L.ora_plan.restype = i32
        _lib = L
    return _lib


def num_threads() -> int:
    return int(lib().ora_num_threads())


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _i32(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x), dtype=np.int32)


def _f32(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().float().numpy()
    return np.ascontiguousarray(np.asarray(x), dtype=np.float32)


def _f64(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x), dtype=np.float64)


def _pool(t: torch.Tensor):
    """A CPU contiguous pool tensor and its dtype code (raw storage is read by C)."""
    t = t.detach().cpu().contiguous()
    return t, DTYPE_CODES[t.dtype]


def _ptr(a) -> int:
    if isinstance(a, torch.Tensor):
        return a.data_ptr()
    return a.ctypes.data


# ---------------------------------------------------------------------------
# public oracle API
# ---------------------------------------------------------------------------

def decode_elements(t: torch.Tensor) -> np.ndarray:
    """Every element of a CPU tensor decoded to f64 by the oracle's own decoder."""
    t, code = _pool(t)
    flat = t.reshape(-1)
    L = lib()
    return np.array([L.ora_decode_element(_ptr(flat), code, i) for i in range(flat.numel())])


def seq_lens(indptr, last_page_len, first_page_offset, page_size) -> list[int]:
    ip, lp, fp = _i32(indptr), _i32(last_page_len), _i32(first_page_offset)
    return [int(lib().ora_seq_len(_ptr(ip), _ptr(lp), _ptr(fp), page_size, r)) for r in range(len(lp))]


def validate_geometry(indptr, last_page_len, first_page_offset, page_size, indices=None,
                      num_pages=0, expect_seq_lens: Sequence[int] | None = None) -> int:
    ip, lp, fp = _i32(indptr), _i32(last_page_len), _i32(first_page_offset)
    batch = len(lp)
    idx = _i32(indices) if indices is not None else None
    sl = np.ascontiguousarray(np.asarray(expect_seq_lens, dtype=np.int64)) if expect_seq_lens is not None else None
    return int(lib().ora_validate_geometry(_ptr(ip), _ptr(lp), _ptr(fp), batch, page_size,
                                           _ptr(idx) if idx is not None else None, int(num_pages),
                                           _ptr(sl) if sl is not None else None))


def resolve_rows(indices, indptr, first_page_offset, page_size, r: int, n: int) -> list[int]:
    """Pool rows (page * page_size + entry) of visible tokens 0..n-1 of request r."""
    idx, ip, fp = _i32(indices), _i32(indptr), _i32(first_page_offset)
    L = lib()
    return [int(L.ora_resolve_row(_ptr(idx), _ptr(ip), _ptr(fp), page_size, r, i)) for i in range(n)]


def _check_table(ip, lp, fp, idx, ps, num_pages, q_batch):
    """Refuse a page table the C routines would read outside of (a test-side mistake, not a result)."""
    if len(ip) != len(lp) + 1 or len(fp) != len(lp) or len(lp) != q_batch:
        raise ValueError("page-table arrays disagree on the batch size")
    if len(ip) and int(ip[-1]) > len(idx):
        raise ValueError(f"indptr[-1] = {int(ip[-1])} exceeds the {len(idx)} indices given")
    code = validate_geometry(ip, lp, fp, ps, idx, num_pages)
    if code != GEOM_OK:
        raise ValueError(f"page table breaks the geometry rules (code {code})")


def attention(q, k_pool, v_pool, indices, indptr, last_page_len, first_page_offset, scale):
    """Decode attention for every (request, query head): (out [B,Hq,D] f64, lse2 [B,Hq] f64)."""
    qf = _f32(q)
    B, Hq, D = qf.shape
    kp, code = _pool(k_pool)
    vp, code_v = _pool(v_pool)
    assert code == code_v and kp.shape == vp.shape
    P, ps, Hkv, Dk = kp.shape
    assert Dk == D
    idx, ip, lp, fp = _i32(indices), _i32(indptr), _i32(last_page_len), _i32(first_page_offset)
    _check_table(ip, lp, fp, idx, ps, P, B)
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    lib().ora_attention(_ptr(qf), _ptr(kp), _ptr(vp), code, _ptr(idx), _ptr(ip), _ptr(lp), _ptr(fp),
                        B, Hq, Hkv, D, ps, float(scale), _ptr(out), _ptr(lse))
    return out, lse


def partials(q, k_pool, v_pool, indices, indptr, last_page_len, first_page_offset, scale,
             pages_per_chunk, request_indices, kv_tile_indices):
    """Per-chunk normalized partials and base-2 LSEs: (v [N,Hq,D] f64, lse2 [N,Hq] f64)."""
    qf = _f32(q)
    B, Hq, D = qf.shape
    kp, code = _pool(k_pool)
    vp, _ = _pool(v_pool)
    P, ps, Hkv, _ = kp.shape
    idx, ip, lp, fp = _i32(indices), _i32(indptr), _i32(last_page_len), _i32(first_page_offset)
    _check_table(ip, lp, fp, idx, ps, P, B)
    ri, ti = _i32(request_indices), _i32(kv_tile_indices)
    N = len(ri)
    out = np.zeros((N, Hq, D), np.float64)
    lse = np.zeros((N, Hq), np.float64)
    lib().ora_partials(_ptr(qf), _ptr(kp), _ptr(vp), code, _ptr(idx), _ptr(ip), _ptr(lp), _ptr(fp),
                       Hq, Hkv, D, ps, int(pages_per_chunk), _ptr(ri), _ptr(ti), N, float(scale),
                       _ptr(out), _ptr(lse))
    return out, lse


def merge(v_in, lse_in, o_indptr):
    """Closed-form merge of attention states grouped by o_indptr: (out [M,H,D], lse2 [M,H])."""
    v, l, oi = _f64(v_in), _f64(lse_in), _i32(o_indptr)
    N, H, D = v.shape
    M = len(oi) - 1
    out = np.zeros((M, H, D), np.float64)
    lse = np.zeros((M, H), np.float64)
    lib().ora_merge(_ptr(v), _ptr(l), _ptr(oi), M, H, D, _ptr(out), _ptr(lse))
    return out, lse


class PlanRef:
    """Result of the oracle plan (linear scan over every chunk size)."""

    def __init__(self, pages_per_chunk, lo, hi, num_chunks, request_indices, kv_tile_indices, o_indptr):
        self.pages_per_chunk = pages_per_chunk
        self.lo = lo
        self.hi = hi
        self.num_chunks = num_chunks
        self.request_indices = request_indices
        self.kv_tile_indices = kv_tile_indices
        self.o_indptr = o_indptr

    @property
    def needs_merge(self) -> bool:
        return self.num_chunks > len(self.o_indptr) - 1


def plan(indptr, num_kv_heads: int, q_groups: int, target_ctas: int, ppc_override: int = 0,
         max_chunks: int = MAX_CHUNKS) -> PlanRef:
    ip = _i32(indptr)
    batch = len(ip) - 1
    cap = int(sum(max(1, int(ip[r + 1] - ip[r])) for r in range(batch)))
    ri = np.zeros(max(cap, 1), np.int32)
    ti = np.zeros(max(cap, 1), np.int32)
    oi = np.zeros(batch + 1, np.int32)
    ppc, lo, hi = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    n = ctypes.c_int64()
    rc = lib().ora_plan(_ptr(ip), batch, num_kv_heads, q_groups, int(target_ctas), int(ppc_override),
                        int(max_chunks), ctypes.addressof(ppc), ctypes.addressof(lo), ctypes.addressof(hi),
                        ctypes.addressof(n), _ptr(ri), _ptr(ti), cap, _ptr(oi))
    if rc != 0:
        raise ValueError(f"oracle plan failed with code {rc}")
    N = int(n.value)
    return PlanRef(int(ppc.value), int(lo.value), int(hi.value), N, ri[:N].copy(), ti[:N].copy(), oi)


def cascade_ref(q, k_pool, v_pool, prefix_indices, suffix_indices, suffix_indptr,
                suffix_last_page_len, scale):
    """Two-level cascade decode of M members sharing a whole-page prefix.

    q: [M, Hq, D].  The prefix pages (all full) are attended once as one
    request whose query heads are the members' heads stacked
    h0 = kv * (M * G) + m * G + g; each member's suffix pages are attended as
    its own request; the two states of member m are merged.  Returns
    (out [M, Hq, D] f64, lse2 [M, Hq] f64).
    """
    qf = torch.as_tensor(_f32(q))
    M, Hq, D = qf.shape
    P, ps, Hkv, _ = k_pool.shape
    G = Hq // Hkv
    # level 0: [M, Hkv, G, D] -> [Hkv, M, G, D], one request with M*Hq heads
    q0 = qf.reshape(M, Hkv, G, D).permute(1, 0, 2, 3).reshape(1, Hkv * M * G, D)
    npre = len(prefix_indices)
    o0, l0 = attention(q0, k_pool, v_pool, prefix_indices, [0, npre], [ps if npre else 0], [0], scale)
    o0 = torch.from_numpy(o0).reshape(Hkv, M, G, D).permute(1, 0, 2, 3).reshape(M, Hq, D)
    l0 = torch.from_numpy(l0).reshape(Hkv, M, G).permute(1, 0, 2).reshape(M, Hq)
    # level 1: each member's private suffix
    o1, l1 = attention(qf, k_pool, v_pool, suffix_indices, suffix_indptr, suffix_last_page_len,
                       [0] * M, scale)
    v_in = torch.stack([o0, torch.from_numpy(o1)], dim=1).reshape(2 * M, Hq, D)
    lse_in = torch.stack([l0, torch.from_numpy(l1)], dim=1).reshape(2 * M, Hq)
    return merge(v_in, lse_in, list(range(0, 2 * M + 1, 2)))


def cascade_detect_ref(indptr, indices, first_page_offset, min_shared_pages: int = 16, min_members: int = 2):
    """Shared-prefix detection (cascade-attention.md, issue #903, the detection paragraphs and table).

    Requests whose window starts mid-page are left out.  The rest are grouped by their first page id;
    a group's shared span is the number of leading page positions on which all its members hold the
    same page id, capped at (pages - 1) for every member (a last page may be partly filled); its score is
    shared * (members - 1), the page reads it removes.  The best-scoring group wins (on a tie, the group
    whose first member comes first in the batch).  It is used only if it has at least `min_members`
    members and `min_shared_pages` shared pages.  Returns (members: sorted request list, shared_pages);
    ([], 0) when nothing qualifies.
    """
    ip = [int(x) for x in _i32(indptr)]
    idx = [int(x) for x in _i32(indices)]
    fp = [int(x) for x in _i32(first_page_offset)]
    B = len(ip) - 1
    groups = {}
    order = []
    for r in range(B):
        pages = ip[r + 1] - ip[r]
        if fp[r] != 0 or pages < 2:
            continue
        key = idx[ip[r]]
        if key not in groups:
            groups[key] = []
            order.append(key)
        groups[key].append(r)
    best, best_score, best_shared = [], -1, 0
    for key in order:
        mem = groups[key]
        if len(mem) < 2:
            continue
        cap = min(ip[r + 1] - ip[r] - 1 for r in mem)
        shared = 0
        while shared < cap and all(idx[ip[r] + shared] == idx[ip[mem[0]] + shared] for r in mem):
            shared += 1
        score = shared * (len(mem) - 1)
        if score > best_score:
            best, best_score, best_shared = mem, score, shared
    if len(best) < max(2, min_members) or best_shared < min_shared_pages:
        return [], 0
    return list(best), best_shared


def selection_rows_ref(block_ids, block_size: int, kv_len: int, request_stride: int):
    """Token rows of a block-sparse selection (sparse-paged-decode.md: "selection_from_blocks expands
    block ids into token rows"; the final-block paragraph: the final block is never scored and is
    appended unconditionally, its live rows only).

    block_ids: [R, topk] ints, each in [0, nb - 1) with nb = ceil(kv_len / block_size).  Request r's
    rows, in this order: for each selected block j (as given), r * request_stride + j * block_size + e
    for e in [0, block_size); then the final block's rows r * request_stride + (nb - 1) * block_size + e
    for e in [0, kv_len - (nb - 1) * block_size).  Returns (indices int32 [R * per_request], per_request).
    """
    ids = [list(map(int, row)) for row in torch.as_tensor(block_ids).reshape(len(block_ids), -1).tolist()]
    nb = (kv_len + block_size - 1) // block_size
    last = kv_len - (nb - 1) * block_size
    out = []
    for r, sel in enumerate(ids):
        base = r * request_stride
        for j in sel:
            if not 0 <= j < nb - 1:
                raise ValueError(f"block id {j} of request {r} outside the scored range [0, {nb - 1})")
            for e in range(block_size):
                out.append(base + j * block_size + e)
        for e in range(last):
            out.append(base + (nb - 1) * block_size + e)
    per_request = len(ids[0]) * block_size + last if ids else 0
    return torch.tensor(out, dtype=torch.int32), per_request


def sparse_csr_ref(num_requests: int, per_request: int):
    """(indptr, last_page_len, first_page_offset) of a token-exact selection: every request lists
    `per_request` one-token pages (sparse-paged-decode.md: the CSR structure follows from the request
    count and the per-request count alone)."""
    indptr = torch.tensor([r * per_request for r in range(num_requests + 1)], dtype=torch.int32)
    ones = torch.tensor([1 if per_request else 0] * num_requests, dtype=torch.int32)
    return indptr, ones, torch.zeros(num_requests, dtype=torch.int32)


def selection_pages_ref(block_ids, block_size: int, kv_len: int, blocks_per_request: int):
    """Block-granular page table of a pool-backed cache whose request r owns pool pages
    [r * blocks_per_request, (r + 1) * blocks_per_request) (sparse-paged-decode.md: feed the selected
    block ids through as indices with the pool's block size as page_size).  The final block goes last so
    that last_page_len can carry its live length.  Returns (indices, indptr, last_page_len,
    first_page_offset)."""
    ids = [list(map(int, row)) for row in torch.as_tensor(block_ids).reshape(len(block_ids), -1).tolist()]
    nb = (kv_len + block_size - 1) // block_size
    last = kv_len - (nb - 1) * block_size
    pages, indptr = [], [0]
    for r, sel in enumerate(ids):
        pages += [r * blocks_per_request + j for j in sel] + [r * blocks_per_request + nb - 1]
        indptr.append(len(pages))
    R = len(ids)
    return (torch.tensor(pages, dtype=torch.int32), torch.tensor(indptr, dtype=torch.int32),
            torch.full((R,), last, dtype=torch.int32), torch.zeros(R, dtype=torch.int32))


def _rows_of(indices, indptr, last_page_len, first_page_offset, page_size, r):
    n = seq_lens(indptr, last_page_len, first_page_offset, page_size)[r]
    return resolve_rows(indices, indptr, first_page_offset, page_size, r, n)


def _attend_extra(qr, qer, K, Ke, V, scale):
    """qr [H, D], qer [H, E], K [n, D], Ke [n, E], V [n, D] (f64) -> out [H, D], lse2 [H]."""
    H = qr.shape[0]
    if K.shape[0] == 0:
        return np.zeros((H, V.shape[1])), np.full(H, -np.inf)
    s = scale * (qr @ K.T + qer @ Ke.T)                   # [H, n], natural-log units
    m = s.max(axis=1, keepdims=True)
    w = np.exp(s - m)
    tot = w.sum(axis=1, keepdims=True)
    return (w / tot) @ V, (m[:, 0] + np.log(tot[:, 0])) / np.log(2.0)


def attention_extra(q, q_extra, k_pool, k_extra_pool, v_pool, dim: int, indices, indptr, last_page_len,
                    first_page_offset, scale):
    """Decode attention with a second K stream, every (request, query head): (out [B,Hq,dim], lse2 [B,Hq]).

    Pools are [P, page_size, Hkv, width] tensors (width >= the dims used: a row's first `dim` elements are
    its K (and, for v_pool, V) part; k_extra_pool's full width is the extra part).  Query head h reads KV
    head h // (Hq / Hkv)."""
    qf = torch.as_tensor(q).double().numpy()
    qe = torch.as_tensor(q_extra).double().numpy()
    B, Hq, D = qf.shape
    assert D == dim
    P, ps, Hkv, _ = k_pool.shape
    G = Hq // Hkv
    kd = k_pool.reshape(P * ps, Hkv, -1)
    ked = k_extra_pool.reshape(P * ps, Hkv, -1)
    vd = v_pool.reshape(P * ps, Hkv, -1)
    out = np.zeros((B, Hq, dim))
    lse = np.zeros((B, Hq))
    ip, lp, fp = _i32(indptr), _i32(last_page_len), _i32(first_page_offset)
    _check_table(ip, lp, fp, _i32(indices), ps, P, B)
    for r in range(B):
        rows = _rows_of(indices, indptr, last_page_len, first_page_offset, ps, r)
        for kvh in range(Hkv):
            K = kd[rows, kvh, :dim].double().numpy()
            Ke = ked[rows, kvh, :].double().numpy()
            V = vd[rows, kvh, :dim].double().numpy()
            hs = slice(kvh * G, (kvh + 1) * G)
            out[r, hs], lse[r, hs] = _attend_extra(qf[r, hs], qe[r, hs], K, Ke, V, scale)
    return out, lse


def partials_extra(q, q_extra, k_pool, k_extra_pool, v_pool, dim: int, indices, indptr, last_page_len,
                   first_page_offset, scale, pages_per_chunk, request_indices, kv_tile_indices):
    """Per-chunk normalized partials and lse2 of the second-K-stream decode.  Chunk (r, k) covers page
    slots [k*ppc, min((k+1)*ppc, pages_r)), i.e. visible tokens [max(0, k*ppc*ps - fpo), min(seq_len,
    (k+1)*ppc*ps - fpo))."""
    qf = torch.as_tensor(q).double().numpy()
    qe = torch.as_tensor(q_extra).double().numpy()
    B, Hq, D = qf.shape
    P, ps, Hkv, _ = k_pool.shape
    G = Hq // Hkv
    kd = k_pool.reshape(P * ps, Hkv, -1)
    ked = k_extra_pool.reshape(P * ps, Hkv, -1)
    vd = v_pool.reshape(P * ps, Hkv, -1)
    ri, ti = _i32(request_indices), _i32(kv_tile_indices)
    fpo = _i32(first_page_offset)
    N = len(ri)
    out = np.zeros((N, Hq, dim))
    lse = np.zeros((N, Hq))
    rows_of = {}
    for c in range(N):
        r, k = int(ri[c]), int(ti[c])
        if r not in rows_of:
            rows_of[r] = _rows_of(indices, indptr, last_page_len, first_page_offset, ps, r)
        rows = rows_of[r]
        t0 = max(0, k * pages_per_chunk * ps - int(fpo[r]))
        t1 = min(len(rows), (k + 1) * pages_per_chunk * ps - int(fpo[r]))
        sel = rows[t0:t1] if t1 > t0 else []
        for kvh in range(Hkv):
            K = kd[sel, kvh, :dim].double().numpy()
            Ke = ked[sel, kvh, :].double().numpy()
            V = vd[sel, kvh, :dim].double().numpy()
            hs = slice(kvh * G, (kvh + 1) * G)
            out[c, hs], lse[c, hs] = _attend_extra(qf[r, hs], qe[r, hs], K, Ke, V, scale)
    return out, lse
