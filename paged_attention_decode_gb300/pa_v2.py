"""Thin ctypes binding of libpa_v2.so (include/pa_v2.h) with the same call names.

Argument marshalling only: every step of the decode path runs in the library's
kernels.  PyTorch provides device memory and streams.  There is no fallback:
if the library is missing or a call fails, a ``PaError`` is raised.

A decode step is ``pa_v2_plan`` (host, cached across steps), then
``pa_v2_decode_partial`` and, when ``plan.needs_merge``, ``pa_merge_states``
(issue #898 "Fused paged-attention decode v2: CSR page table, cross-CTA
split-KV, and variable-length merge kernels", design pieces 2-4).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa_v2.so")

PA_OK, PA_EINVAL, PA_EGEOMETRY, PA_ECAPACITY, PA_EUNSUPPORTED, PA_ECUDA, PA_EOOB = 0, -1, -2, -3, -4, -5, -6
PA_F32, PA_F16, PA_BF16 = 0, 1, 2
PA_V2_MAX_CHUNKS = 65535
DEVICE_BAD_REQUEST, DEVICE_BAD_SLOT, DEVICE_BAD_PAGE, DEVICE_BAD_INDPTR, DEVICE_WAIT_TIMEOUT = 1, 2, 4, 8, 16
DEVICE_BAD_BLOCK = 32

KV_DTYPES = {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16}

# Exported symbols of the C ABI (the header's declarations).
ABI_SYMBOLS = ("pa_v2_q_heads_per_cta", "pa_v2_default_target_ctas", "pa_v2_plan", "pa_v2_plan_matches",
               "pa_v2_decode_partial", "pa_v2_decode", "pa_v2_decode_noalloc", "pa_merge_states",
               "pa_v2_cascade_detect", "pa_v2_cascade_split", "pa_selection_rows_per_request", "pa_sparse_csr",
               "pa_selection_from_blocks", "pa_v2_host_io_layout", "pa_v2_decode_host",
               "pa_v2_decode_partial_extra", "pa_v2_selftest_wait", "pa_v2_host_graph_create",
               "pa_v2_host_graph_run", "pa_v2_host_graph_destroy", "pa_v2_decode_host_mapped",
               "pa_v2_host_graph_create_mapped", "pa_v2_wave_fit_pages_per_chunk",
               "pa_v2_balanced_pages_per_chunk", "pa_v2_cascade_plan", "pa_v2_cascade_decode",
               "pa_status_from_device", "pa_status_string", "pa_version")
NOALLOC_SCRATCH_BYTES = 8 << 20


class CascadeLevelStruct(ctypes.Structure):
    """Mirror of pa_v2_cascade_level_t (device pointers of one cascade level)."""

    _fields_ = [("indices", ctypes.c_void_p), ("num_indices", ctypes.c_int64), ("indptr", ctypes.c_void_p),
                ("last_page_len", ctypes.c_void_p), ("first_page_offset", ctypes.c_void_p),
                ("request_indices", ctypes.c_void_p), ("kv_tile_indices", ctypes.c_void_p),
                ("member_rows", ctypes.c_void_p), ("part_rows", ctypes.c_void_p)]


class PaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {pa_status_string(status)} ({status})")


class PlanStruct(ctypes.Structure):
    """Mirror of pa_v2_plan_t."""

    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "num_qo_heads", "num_kv_heads", "head_dim", "page_size", "kv_dtype", "q_heads_per_cta",
        "q_groups", "pages_per_chunk", "lo_pages_per_chunk", "hi_pages_per_chunk", "num_chunks",
        "needs_merge", "target_ctas", "total_ctas", "kernel", "stack_members", "out_row_step")] + [
        ("num_indices", ctypes.c_int64), ("workspace_v_bytes", ctypes.c_int64),
        ("workspace_lse_bytes", ctypes.c_int64), ("counter_bytes", ctypes.c_int64),
        ("geometry_hash", ctypes.c_uint64)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libpa_v2.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with paged_attention_decode_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        PP = ctypes.POINTER(PlanStruct)
        L.pa_v2_q_heads_per_cta.argtypes = [i32, i32, i32]
        L.pa_v2_q_heads_per_cta.restype = i32
        L.pa_v2_default_target_ctas.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(i32)]
        L.pa_v2_default_target_ctas.restype = i32
        L.pa_v2_plan.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, P, P, i32, P, PP]
        L.pa_v2_plan.restype = i32
        L.pa_v2_plan_matches.argtypes = [PP, P, P, P, i32]
        L.pa_v2_plan_matches.restype = i32
        L.pa_v2_decode_partial.argtypes = [PP, P, P, P, i32, i64, P, i64, P, P, P, P, P, f32, P, P, P, P]
        L.pa_v2_decode_partial.restype = i32
        L.pa_v2_decode.argtypes = [PP, P, P, P, i32, i64, P, i64, P, P, P, P, P, P, f32, P, P, P, P, P, P, P, P, P]
        L.pa_v2_cascade_detect.argtypes = [P, P, P, i32, i32, i32, P, P, P]
        L.pa_v2_cascade_detect.restype = i32
        L.pa_v2_cascade_split.argtypes = [P, P, P, P, i32, P, i32, P, P, P, P, P, P, P, P]
        L.pa_v2_cascade_split.restype = i32
        L.pa_v2_cascade_plan.argtypes = [i32, i32, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, P, P, i32, P,
                                         P, P, i32, P, P, P, P, PP, PP]
        L.pa_v2_cascade_plan.restype = i32
        CL = ctypes.POINTER(CascadeLevelStruct)
        L.pa_v2_cascade_decode.argtypes = [PP, PP, CL, CL, P, P, P, i32, i64, f32, P, P, i32, P, i32, P, P, P, P]
        L.pa_v2_cascade_decode.restype = i32
        L.pa_v2_decode.restype = i32
        L.pa_v2_decode_noalloc.argtypes = [PP, P, P, P, i32, i64, P, i64, P, P, P, P, P, P, f32, P, P, P, P]
        L.pa_v2_decode_noalloc.restype = i32
        L.pa_merge_states.argtypes = [P, P, P, i32, i32, i32, i32, P, P, P, P]
        L.pa_merge_states.restype = i32
        L.pa_v2_host_io_layout.argtypes = [PP, ctypes.POINTER(i64), ctypes.POINTER(i64), ctypes.POINTER(i64)]
        L.pa_v2_host_io_layout.restype = i32
        L.pa_v2_decode_host.argtypes = [PP, P, P, P, P, P, i32, i64, P, P, P, f32, P, P, P]
        L.pa_v2_decode_host.restype = i32
        L.pa_v2_decode_partial_extra.argtypes = [PP, P, P, P, i64, P, i64, P, i64, i32, i32, i64, P, i64, P, P, P,
                                                 P, P, f32, P, P, P, P]
        L.pa_v2_decode_partial_extra.restype = i32
        L.pa_v2_selftest_wait.argtypes = [P, P, i64, P]
        L.pa_v2_selftest_wait.restype = i32
        L.pa_v2_host_graph_create.argtypes = [PP, P, P, P, P, P, i32, i64, P, P, P, f32, P, P, P]
        L.pa_v2_host_graph_create.restype = i32
        L.pa_v2_decode_host_mapped.argtypes = [PP, P, P, P, P, i32, i64, P, P, P, f32, P, P, P]
        L.pa_v2_decode_host_mapped.restype = i32
        L.pa_v2_host_graph_create_mapped.argtypes = [PP, P, P, P, P, i32, i64, P, P, P, f32, P, P, P]
        L.pa_v2_host_graph_create_mapped.restype = i32
        L.pa_v2_host_graph_run.argtypes = [P, P]
        L.pa_v2_host_graph_run.restype = i32
        L.pa_v2_host_graph_destroy.argtypes = [P]
        L.pa_v2_host_graph_destroy.restype = None
        L.pa_v2_wave_fit_pages_per_chunk.argtypes = [P, i32, i32, i32]
        L.pa_v2_wave_fit_pages_per_chunk.restype = i32
        L.pa_v2_balanced_pages_per_chunk.argtypes = [P, i32, i32, i32]
        L.pa_v2_balanced_pages_per_chunk.restype = i32
        L.pa_selection_rows_per_request.argtypes = [i32, i32, i32]
        L.pa_selection_rows_per_request.restype = i64
        L.pa_sparse_csr.argtypes = [i32, i64, P, P, P]
        L.pa_sparse_csr.restype = i32
        L.pa_selection_from_blocks.argtypes = [P, i32, i32, i32, i32, i64, P, P, P]
        L.pa_selection_from_blocks.restype = i32
        L.pa_status_from_device.argtypes = [i32]
        L.pa_status_from_device.restype = i32
        L.pa_status_string.argtypes = [i32]
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_version.restype = ctypes.c_char_p
        _lib = L
    return _lib


def pa_status_string(status: int) -> str:
    return lib().pa_status_string(int(status)).decode()


def pa_status_from_device(word: int) -> int:
    return int(lib().pa_status_from_device(int(word)))


def pa_version() -> str:
    return lib().pa_version().decode()


def pa_v2_q_heads_per_cta(group_size: int, head_dim: int, kv_dtype: int) -> int:
    return int(lib().pa_v2_q_heads_per_cta(group_size, head_dim, kv_dtype))


def pa_v2_default_target_ctas(num_qo_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
                              kv_dtype: int, device: int | None = None) -> int:
    dev = torch.cuda.current_device() if device is None else device
    out = ctypes.c_int32()
    rc = lib().pa_v2_default_target_ctas(dev, num_qo_heads, num_kv_heads, head_dim, page_size, kv_dtype,
                                         ctypes.byref(out))
    if rc != PA_OK:
        raise PaError(rc, "pa_v2_default_target_ctas")
    return int(out.value)


def _host_i32(x) -> torch.Tensor:
    t = torch.as_tensor(x)
    return t.detach().to("cpu", torch.int32).contiguous()


@dataclass
class Plan:
    """A plan plus its chunk index arrays (host copies; device copies made on demand)."""

    struct: PlanStruct
    request_indices: torch.Tensor
    kv_tile_indices: torch.Tensor
    o_indptr: torch.Tensor
    _dev: dict | None = None

    def __getattr__(self, name):
        if name.startswith("_") or name in ("struct",):
            raise AttributeError(name)
        return getattr(self.struct, name)

    def device_counters(self, device) -> torch.Tensor:
        """Zeroed int32 ticket counters for pa_v2_decode on `device`, allocated once (the kernel leaves
        them zero after every successful launch)."""
        key = "counters:" + str(torch.device(device))
        if self._dev is None:
            self._dev = {}
        if key not in self._dev:
            self._dev[key] = torch.zeros(max(1, self.struct.counter_bytes // 4), dtype=torch.int32, device=device)
        return self._dev[key]

    def device_arrays(self, device) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
        """(request_indices, kv_tile_indices, o_indptr) on `device`, uploaded once."""
        key = str(torch.device(device))
        if self._dev is None:
            self._dev = {}
        if key not in self._dev:
            self._dev[key] = tuple(t.to(device) for t in (self.request_indices, self.kv_tile_indices, self.o_indptr))
        return self._dev[key]


def pa_v2_plan(indptr, last_page_len, first_page_offset, page_size: int, num_qo_heads: int, num_kv_heads: int,
               head_dim: int, kv_dtype: int, target_ctas: int = 0, pages_per_chunk_override: int = 0,
               seq_lens=None) -> Plan:
    """Host plan (pa_v2_plan).  Inputs are host arrays (any int sequence / CPU tensor)."""
    ip, lp, fp = _host_i32(indptr), _host_i32(last_page_len), _host_i32(first_page_offset)
    batch = lp.numel()
    sl = _host_i32(seq_lens) if seq_lens is not None else None
    pages = (ip[1:] - ip[:-1]).clamp(min=1) if batch else ip[:0]
    cap = int(pages.sum()) if batch else 0
    ri = torch.zeros(max(cap, 1), dtype=torch.int32)
    ti = torch.zeros(max(cap, 1), dtype=torch.int32)
    oi = torch.zeros(batch + 1, dtype=torch.int32)
    st = PlanStruct()
    rc = lib().pa_v2_plan(ip.data_ptr(), lp.data_ptr(), fp.data_ptr(), sl.data_ptr() if sl is not None else None,
                          batch, page_size, num_qo_heads, num_kv_heads, head_dim, kv_dtype, target_ctas,
                          pages_per_chunk_override, ri.data_ptr(), ti.data_ptr(), cap, oi.data_ptr(),
                          ctypes.byref(st))
    if rc != PA_OK:
        raise PaError(rc, "pa_v2_plan")
    n = st.num_chunks
    return Plan(st, ri[:n].clone(), ti[:n].clone(), oi)


def pa_v2_plan_matches(plan: Plan, indptr, last_page_len, first_page_offset) -> bool:
    ip, lp, fp = _host_i32(indptr), _host_i32(last_page_len), _host_i32(first_page_offset)
    return bool(lib().pa_v2_plan_matches(ctypes.byref(plan.struct), ip.data_ptr(), lp.data_ptr(), fp.data_ptr(),
                                         lp.numel()))


def _dev_ptr(t: torch.Tensor | None, name: str, dtype=None) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _out_ptr(t: torch.Tensor, name: str, s: PlanStruct, per_row: int) -> int:
    """Pointer of a final-output tensor whose rows may be `out_row_step` rows apart: either contiguous,
    or a view whose leading dimension has stride out_row_step * per_row elements (rows interleaved with
    another decode's rows for one pa_merge_states)."""
    if not t.is_cuda or t.dtype != torch.float32:
        raise ValueError(f"{name} must be a float32 CUDA tensor")
    if t.is_contiguous():
        return t.data_ptr()
    inner = t[0] if t.dim() > 1 else t
    if t.dim() < 2 or not inner.is_contiguous() or t.stride(0) != s.out_row_step * per_row:
        raise ValueError(f"{name} must be contiguous, or rows {s.out_row_step} x {per_row} elements apart")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def pa_v2_decode_partial(plan: Plan, q, k_pool, v_pool, indices, indptr, last_page_len, first_page_offset,
                         sm_scale: float, v_out=None, lse2_out=None, status=None, stream=None,
                         request_indices=None, kv_tile_indices=None):
    """Partial kernel (pa_v2_decode_partial).  Device tensors; returns (v_out [N,Hq,D], lse2_out [N,Hq])."""
    s = plan.struct
    dev = q.device
    if request_indices is None or kv_tile_indices is None:
        request_indices, kv_tile_indices, _ = plan.device_arrays(dev)
    if k_pool.dtype not in KV_DTYPES or v_pool.dtype != k_pool.dtype or k_pool.shape != v_pool.shape:
        raise ValueError("k_pool and v_pool must share one of float32/float16/bfloat16 and a shape")
    if k_pool.dim() != 4 or tuple(k_pool.shape[1:]) != (s.page_size, s.num_kv_heads, s.head_dim):
        raise ValueError(f"pools must be [P, {s.page_size}, {s.num_kv_heads}, {s.head_dim}]")
    if v_out is None:
        v_out = torch.empty(max(s.num_chunks, 1), s.num_qo_heads, s.head_dim, device=dev, dtype=torch.float32)
    if lse2_out is None:
        lse2_out = torch.empty(max(s.num_chunks, 1), s.num_qo_heads, device=dev, dtype=torch.float32)
    rc = lib().pa_v2_decode_partial(
        ctypes.byref(s), _dev_ptr(q, "q", torch.float32), _dev_ptr(k_pool, "k_pool"), _dev_ptr(v_pool, "v_pool"),
        KV_DTYPES[k_pool.dtype], k_pool.shape[0], _dev_ptr(indices, "indices", torch.int32), indices.numel(),
        _dev_ptr(indptr, "indptr", torch.int32), _dev_ptr(last_page_len, "last_page_len", torch.int32),
        _dev_ptr(first_page_offset, "first_page_offset", torch.int32),
        _dev_ptr(request_indices, "request_indices", torch.int32),
        _dev_ptr(kv_tile_indices, "kv_tile_indices", torch.int32), float(sm_scale),
        _dev_ptr(v_out, "v_out", torch.float32), _dev_ptr(lse2_out, "lse2_out", torch.float32),
        _dev_ptr(status, "status", torch.int32), _stream(stream))
    if rc != PA_OK:
        raise PaError(rc, "pa_v2_decode_partial")
    return v_out, lse2_out


def pa_merge_states(v_in, lse2_in, o_indptr, num_rows_out: int, v_out=None, lse2_out=None, status=None,
                    stream=None):
    """Merge kernel (pa_merge_states).  Device tensors; returns (v_out [M,H,D], lse2_out [M,H])."""
    N, H, D = v_in.shape
    dev = v_in.device
    if v_out is None:
        v_out = torch.empty(num_rows_out, H, D, device=dev, dtype=torch.float32)
    if lse2_out is None:
        lse2_out = torch.empty(num_rows_out, H, device=dev, dtype=torch.float32)
    rc = lib().pa_merge_states(_dev_ptr(v_in, "v_in", torch.float32), _dev_ptr(lse2_in, "lse2_in", torch.float32),
                               _dev_ptr(o_indptr, "o_indptr", torch.int32), num_rows_out, N, H, D,
                               _dev_ptr(v_out, "v_out", torch.float32),
                               _dev_ptr(lse2_out, "lse2_out", torch.float32),
                               _dev_ptr(status, "status", torch.int32), _stream(stream))
    if rc != PA_OK:
        raise PaError(rc, "pa_merge_states")
    return v_out, lse2_out


def pa_v2_decode(plan: Plan, q, k_pool, v_pool, indices, indptr, last_page_len, first_page_offset,
                 sm_scale: float, out=None, lse2_out=None, workspace=None, counters=None, status=None, stream=None,
                 request_indices=None, kv_tile_indices=None, o_indptr=None, member_rows=None, out_rows=None):
    """One-launch decode (pa_v2_decode): partial kernel with the merge fused in.

    Returns (out [B, Hq, D] f32, lse2 [B, Hq] f32).  `workspace` = (v, lse) partial buffers sized by the
    plan; `counters` = zeroed int32 [plan.counter_bytes // 4] (the plan keeps one per device by default).
    """
    s = plan.struct
    dev = q.device
    ri, ti, oi = plan.device_arrays(dev)
    ri = ri if request_indices is None else request_indices
    ti = ti if kv_tile_indices is None else kv_tile_indices
    oi = oi if o_indptr is None else o_indptr
    if counters is None:
        counters = plan.device_counters(dev)
    wv, wl = workspace if workspace is not None else (None, None)
    if wv is None:
        wv = torch.empty(max(s.num_chunks, 1), s.num_qo_heads, s.head_dim, device=dev, dtype=torch.float32)
    if wl is None:
        wl = torch.empty(max(s.num_chunks, 1), s.num_qo_heads, device=dev, dtype=torch.float32)
    rows = s.batch * s.stack_members        # requests, or members of a stacked (cascade level 0) plan
    heads = s.num_qo_heads // s.stack_members
    if out is None:
        out = torch.empty(max(rows, 1) * s.out_row_step, heads, s.head_dim, device=dev,
                          dtype=torch.float32)[::s.out_row_step]
    if lse2_out is None:
        lse2_out = torch.empty(max(rows, 1) * s.out_row_step, heads, device=dev, dtype=torch.float32)[::s.out_row_step]
    if k_pool.dtype not in KV_DTYPES or v_pool.dtype != k_pool.dtype or k_pool.shape != v_pool.shape:
        raise ValueError("k_pool and v_pool must share one of float32/float16/bfloat16 and a shape")
    if counters.numel() * 4 < s.counter_bytes:
        raise ValueError("counters too small for the plan")
    rc = lib().pa_v2_decode(
        ctypes.byref(s), _dev_ptr(q, "q", torch.float32), _dev_ptr(k_pool, "k_pool"), _dev_ptr(v_pool, "v_pool"),
        KV_DTYPES[k_pool.dtype], k_pool.shape[0], _dev_ptr(indices, "indices", torch.int32), indices.numel(),
        _dev_ptr(indptr, "indptr", torch.int32), _dev_ptr(last_page_len, "last_page_len", torch.int32),
        _dev_ptr(first_page_offset, "first_page_offset", torch.int32),
        _dev_ptr(ri, "request_indices", torch.int32), _dev_ptr(ti, "kv_tile_indices", torch.int32),
        _dev_ptr(oi, "o_indptr", torch.int32), float(sm_scale), _dev_ptr(wv, "workspace_v", torch.float32),
        _dev_ptr(wl, "workspace_lse", torch.float32), _dev_ptr(counters, "counters", torch.int32),
        _out_ptr(out, "out", s, heads * s.head_dim) if out_rows is None else _dev_ptr(out, "out", torch.float32),
        _out_ptr(lse2_out, "lse2_out", s, heads) if out_rows is None else _dev_ptr(lse2_out, "lse2_out", torch.float32),
        _dev_ptr(member_rows, "member_rows", torch.int32), _dev_ptr(out_rows, "out_rows", torch.int32),
        _dev_ptr(status, "status", torch.int32), _stream(stream))
    if rc != PA_OK:
        raise PaError(rc, "pa_v2_decode")
    return (out[:rows], lse2_out[:rows]) if out_rows is None else (out, lse2_out)


def pa_v2_cascade_detect(indptr, indices, first_page_offset, min_shared_pages: int = 16, min_members: int = 2):
    """Shared-prefix detection (pa_v2_cascade_detect); host arrays.  Returns (member flags [B], shared pages)."""
    ip, idx, fp = _host_i32(indptr), _host_i32(indices), _host_i32(first_page_offset)
    B = fp.numel()
    flags = torch.zeros(max(B, 1), dtype=torch.int32)
    nm, sh = ctypes.c_int32(), ctypes.c_int32()
    rc = lib().pa_v2_cascade_detect(ip.data_ptr(), idx.data_ptr() if idx.numel() else None, fp.data_ptr(), B,
                                    min_shared_pages, min_members, flags.data_ptr(), ctypes.byref(nm),
                                    ctypes.byref(sh))
    if rc != PA_OK:
        raise PaError(rc, "pa_v2_cascade_detect")
    return flags[:B], int(sh.value)


def pa_v2_cascade_split(indptr, indices, last_page_len, first_page_offset, member_of, shared_pages: int):
    """Level-1 table and row maps of a cascade batch (pa_v2_cascade_split); host arrays in and out."""
    ip, idx, lp, fp, mo = (_host_i32(x) for x in (indptr, indices, last_page_len, first_page_offset, member_of))
    B = lp.numel()
    M = int(mo.sum())
    l1_ip = torch.zeros(B + 1, dtype=torch.int32)
    l1_idx = torch.zeros(max(1, idx.numel() - M * shared_pages), dtype=torch.int32)
    l1_lp = torch.zeros(max(B, 1), dtype=torch.int32)
    l1_fp = torch.zeros(max(B, 1), dtype=torch.int32)
    mrows = torch.zeros(max(M, 1), dtype=torch.int32)
    l0_rows = torch.zeros(max(M, 1), dtype=torch.int32)
    l1_rows = torch.zeros(max(B, 1), dtype=torch.int32)
    m_ip = torch.zeros(B + 1, dtype=torch.int32)
    rc = lib().pa_v2_cascade_split(ip.data_ptr(), idx.data_ptr(), lp.data_ptr(), fp.data_ptr(), B, mo.data_ptr(),
                                   shared_pages, l1_ip.data_ptr(), l1_idx.data_ptr(), l1_lp.data_ptr(),
                                   l1_fp.data_ptr(), mrows.data_ptr(), l0_rows.data_ptr(), l1_rows.data_ptr(),
                                   m_ip.data_ptr())
    if rc != PA_OK:
        raise PaError(rc, "pa_v2_cascade_split")
    n1 = int(l1_ip[-1])
    return {"l1_indptr": l1_ip, "l1_indices": l1_idx[:n1], "l1_last_page_len": l1_lp[:B],
            "l1_first_page_offset": l1_fp[:B], "member_rows": mrows[:M], "l0_out_rows": l0_rows[:M],
            "l1_out_rows": l1_rows[:B], "merge_indptr": m_ip}


@dataclass
class CascadePlans:
    """Both cascade levels' plans and the merge input they share (pa_v2_cascade_plan); host arrays."""

    level0: Plan
    level1: Plan
    l0_part_rows: torch.Tensor   # [members]
    l1_part_rows: torch.Tensor   # [l1_batch]
    merge_indptr: torch.Tensor   # [l1_batch + 1]

    @property
    def merge_rows(self) -> int:
        return int(self.merge_indptr[-1])


def pa_v2_cascade_plan(members: int, shared_pages: int, l1_indptr, l1_last_page_len, l1_first_page_offset,
                       page_size: int, num_qo_heads: int, num_kv_heads: int, head_dim: int, kv_dtype: int,
                       wave_ctas: int, l1_seq_lens=None, member_requests=None) -> CascadePlans:
    """Plans of both cascade levels for one launch, and the merge layout (pa_v2_cascade_plan); host arrays."""
    ip, lp, fp = _host_i32(l1_indptr), _host_i32(l1_last_page_len), _host_i32(l1_first_page_offset)
    B = lp.numel()
    sl = _host_i32(l1_seq_lens) if l1_seq_lens is not None else None
    mr = _host_i32(member_requests) if member_requests is not None else None
    cap1 = int((ip[1:] - ip[:-1]).clamp(min=1).sum()) if B else 1
    cap0 = max(1, int(shared_pages))
    r0, t0, o0 = (torch.zeros(cap0, dtype=torch.int32), torch.zeros(cap0, dtype=torch.int32),
                  torch.zeros(2, dtype=torch.int32))
    r1, t1, o1 = (torch.zeros(max(cap1, 1), dtype=torch.int32), torch.zeros(max(cap1, 1), dtype=torch.int32),
                  torch.zeros(B + 1, dtype=torch.int32))
    pr0, pr1 = torch.zeros(max(members, 1), dtype=torch.int32), torch.zeros(max(B, 1), dtype=torch.int32)
    mi = torch.zeros(B + 1, dtype=torch.int32)
    s0, s1 = PlanStruct(), PlanStruct()
    rc = lib().pa_v2_cascade_plan(members, shared_pages, ip.data_ptr(), lp.data_ptr() if B else None,
                                  fp.data_ptr() if B else None, sl.data_ptr() if sl is not None else None, B,
                                  mr.data_ptr() if mr is not None else None, page_size, num_qo_heads, num_kv_heads,
                                  head_dim, kv_dtype, wave_ctas, r0.data_ptr(), t0.data_ptr(), cap0, o0.data_ptr(),
                                  r1.data_ptr(), t1.data_ptr(), max(cap1, 1), o1.data_ptr(), pr0.data_ptr(),
                                  pr1.data_ptr(), mi.data_ptr(), ctypes.byref(s0), ctypes.byref(s1))
    if rc != PA_OK:
        raise PaError(rc, "pa_v2_cascade_plan")
    return CascadePlans(Plan(s0, r0[:s0.num_chunks].clone(), t0[:s0.num_chunks].clone(), o0),
                        Plan(s1, r1[:s1.num_chunks].clone(), t1[:s1.num_chunks].clone(), o1),
                        pr0[:members].clone(), pr1[:B].clone(), mi)


def cascade_level(plan: Plan, indices, indptr, last_page_len, first_page_offset, part_rows,
                  member_rows=None) -> CascadeLevelStruct:
    """A pa_v2_cascade_level_t for `plan` (device tensors; the plan's chunk arrays are its own device
    copies, kept alive by the struct)."""
    dev = indices.device
    ri, ti, _ = plan.device_arrays(dev)
    lv = CascadeLevelStruct()
    lv.indices = _dev_ptr(indices, "indices", torch.int32)
    lv.num_indices = indices.numel()
    lv.indptr = _dev_ptr(indptr, "indptr", torch.int32)
    lv.last_page_len = _dev_ptr(last_page_len, "last_page_len", torch.int32)
    lv.first_page_offset = _dev_ptr(first_page_offset, "first_page_offset", torch.int32)
    lv.request_indices = _dev_ptr(ri, "request_indices", torch.int32)
    lv.kv_tile_indices = _dev_ptr(ti, "kv_tile_indices", torch.int32)
    lv.member_rows = _dev_ptr(member_rows, "member_rows", torch.int32)
    lv.part_rows = _dev_ptr(part_rows, "part_rows", torch.int32)
    lv._keep = (ri, ti, part_rows, member_rows)
    return lv


def pa_v2_cascade_decode(cps: CascadePlans, level0: CascadeLevelStruct, level1: CascadeLevelStruct, q, k_pool,
                         v_pool, sm_scale: float, merge_v, merge_lse, merge_indptr, out=None, lse2_out=None,
                         status=None, stream=None):
    """Both cascade levels in one launch writing one merge input, then the merge (pa_v2_cascade_decode).
    Returns (out [B, Hq, D], lse2 [B, Hq]), B = the level-1 batch."""
    p1 = cps.level1.struct
    H, D, B = p1.num_qo_heads, p1.head_dim, p1.batch
    dev = q.device
    if out is None:
        out = torch.empty(max(B, 1), H, D, device=dev, dtype=torch.float32)
    if lse2_out is None:
        lse2_out = torch.empty(max(B, 1), H, device=dev, dtype=torch.float32)
    if tuple(merge_v.shape) != (cps.merge_rows, H, D) or tuple(merge_lse.shape) != (cps.merge_rows, H):
        raise ValueError(f"merge_v / merge_lse must be [{cps.merge_rows}, {H}, {D}] / [{cps.merge_rows}, {H}]")
    if k_pool.dtype not in KV_DTYPES or v_pool.dtype != k_pool.dtype or k_pool.shape != v_pool.shape:
        raise ValueError("k_pool and v_pool must share one of float32/float16/bfloat16 and a shape")
    rc = lib().pa_v2_cascade_decode(
        ctypes.byref(cps.level0.struct), ctypes.byref(p1), ctypes.byref(level0), ctypes.byref(level1),
        _dev_ptr(q, "q", torch.float32), _dev_ptr(k_pool, "k_pool"), _dev_ptr(v_pool, "v_pool"),
        KV_DTYPES[k_pool.dtype], k_pool.shape[0], float(sm_scale), _dev_ptr(merge_v, "merge_v", torch.float32),
        _dev_ptr(merge_lse, "merge_lse", torch.float32), cps.merge_rows,
        _dev_ptr(merge_indptr, "merge_indptr", torch.int32), B, _dev_ptr(out, "out", torch.float32),
        _dev_ptr(lse2_out, "lse2_out", torch.float32), _dev_ptr(status, "status", torch.int32), _stream(stream))
    if rc != PA_OK:
        raise PaError(rc, "pa_v2_cascade_decode")
    return out[:B], lse2_out[:B]


def pa_v2_decode_noalloc(plan: Plan, q, k_pool, v_pool, indices, indptr, last_page_len, first_page_offset,
                         sm_scale: float, out=None, lse2_out=None, status=None, stream=None):
    """pa_v2_decode for callers that cannot allocate device memory (pa_v2_decode_noalloc).

    The partial workspace and the ticket counters come from the library's own fixed device array
    (NOALLOC_SCRATCH_BYTES per GPU); the caller supplies every input and output.  Calls on one device
    share that array, so keep them ordered on one stream.  Outputs are laid out as pa_v2_decode's with
    no row maps: request r (member m of a stacked plan) at row r * out_row_step (m * out_row_step).
    Returns (out [rows, heads, D], lse2 [rows, heads]), rows = batch * stack_members.
    """
    s = plan.struct
    dev = q.device
    ri, ti, oi = plan.device_arrays(dev)
    rows = s.batch * s.stack_members        # requests, or members of a stacked (cascade level 0) plan
    heads = s.num_qo_heads // s.stack_members
    if out is None:
        out = torch.empty(max(rows, 1) * s.out_row_step, heads, s.head_dim, device=dev,
                          dtype=torch.float32)[::s.out_row_step]
    if lse2_out is None:
        lse2_out = torch.empty(max(rows, 1) * s.out_row_step, heads, device=dev, dtype=torch.float32)[::s.out_row_step]
    if out.shape[0] < rows or tuple(out.shape[1:]) != (heads, s.head_dim):
        raise ValueError(f"out must hold [{rows}, {heads}, {s.head_dim}]")
    if lse2_out.shape[0] < rows or tuple(lse2_out.shape[1:]) != (heads,):
        raise ValueError(f"lse2_out must hold [{rows}, {heads}]")
    if k_pool.dtype not in KV_DTYPES or v_pool.dtype != k_pool.dtype or k_pool.shape != v_pool.shape:
        raise ValueError("k_pool and v_pool must share one of float32/float16/bfloat16 and a shape")
    rc = lib().pa_v2_decode_noalloc(
        ctypes.byref(s), _dev_ptr(q, "q", torch.float32), _dev_ptr(k_pool, "k_pool"), _dev_ptr(v_pool, "v_pool"),
        KV_DTYPES[k_pool.dtype], k_pool.shape[0], _dev_ptr(indices, "indices", torch.int32), indices.numel(),
        _dev_ptr(indptr, "indptr", torch.int32), _dev_ptr(last_page_len, "last_page_len", torch.int32),
        _dev_ptr(first_page_offset, "first_page_offset", torch.int32),
        _dev_ptr(ri, "request_indices", torch.int32), _dev_ptr(ti, "kv_tile_indices", torch.int32),
        _dev_ptr(oi, "o_indptr", torch.int32), float(sm_scale), _out_ptr(out, "out", s, heads * s.head_dim),
        _out_ptr(lse2_out, "lse2_out", s, heads), _dev_ptr(status, "status", torch.int32), _stream(stream))
    if rc != PA_OK:
        raise PaError(rc, "pa_v2_decode_noalloc")
    return out[:rows], lse2_out[:rows]


def decode(plan: Plan, q, k_pool, v_pool, indices, indptr, last_page_len, first_page_offset, sm_scale: float,
           out=None, lse2=None, workspace=None, status=None, stream=None):
    """One decode step: the partial launch, then the merge launch when the plan needs one.

    Returns (out [B, Hq, D] f32, lse2 [B, Hq] f32).  `workspace` may supply the
    (v, lse) partial buffers sized by the plan.
    """
    s = plan.struct
    ri, ti, oi = plan.device_arrays(q.device)
    if not s.needs_merge:
        v, l = pa_v2_decode_partial(plan, q, k_pool, v_pool, indices, indptr, last_page_len, first_page_offset,
                                    sm_scale, out, lse2, status, stream, ri, ti)
        return v[:s.batch], l[:s.batch]
    wv, wl = workspace if workspace is not None else (None, None)
    wv, wl = pa_v2_decode_partial(plan, q, k_pool, v_pool, indices, indptr, last_page_len, first_page_offset,
                                  sm_scale, wv, wl, status, stream, ri, ti)
    return pa_merge_states(wv, wl, oi, s.batch, out, lse2, status, stream)


# ---------------------------------------------------------------------------
# block-sparse selections
# ---------------------------------------------------------------------------

def pa_selection_rows_per_request(topk: int, block_size: int, kv_len: int) -> int:
    """Rows each request's token-exact page table lists (pa_selection_rows_per_request); raises if invalid."""
    n = int(lib().pa_selection_rows_per_request(int(topk), int(block_size), int(kv_len)))
    if n < 0:
        raise PaError(PA_EINVAL, "pa_selection_rows_per_request")
    return n


def pa_sparse_csr(num_requests: int, per_request: int):
    """Host (indptr, last_page_len, first_page_offset) of a token-exact selection (pa_sparse_csr)."""
    ip = torch.empty(num_requests + 1, dtype=torch.int32)
    lp = torch.empty(max(num_requests, 1), dtype=torch.int32)
    fp = torch.empty(max(num_requests, 1), dtype=torch.int32)
    rc = lib().pa_sparse_csr(int(num_requests), int(per_request), ip.data_ptr(), lp.data_ptr(), fp.data_ptr())
    if rc != PA_OK:
        raise PaError(rc, "pa_sparse_csr")
    return ip, lp[:num_requests], fp[:num_requests]


def pa_selection_from_blocks(block_ids, block_size: int, kv_len: int, request_stride: int, indices=None,
                             status=None, stream=None):
    """Token rows of a block-sparse selection (pa_selection_from_blocks).  block_ids: device int32
    [num_requests, topk].  Returns the device int32 indices [num_requests * per_request]."""
    R, topk = block_ids.shape
    per = pa_selection_rows_per_request(topk, block_size, kv_len)
    if indices is None:
        indices = torch.empty(max(1, R * per), dtype=torch.int32, device=block_ids.device)
    if indices.numel() < R * per:
        raise ValueError("indices too small for the selection")
    rc = lib().pa_selection_from_blocks(_dev_ptr(block_ids, "block_ids", torch.int32) if topk else None, R, topk,
                                        int(block_size), int(kv_len), int(request_stride),
                                        _dev_ptr(indices, "indices", torch.int32),
                                        _dev_ptr(status, "status", torch.int32), _stream(stream))
    if rc != PA_OK:
        raise PaError(rc, "pa_selection_from_blocks")
    return indices[:R * per]


# ---------------------------------------------------------------------------
# one step from host buffers
# ---------------------------------------------------------------------------

def pa_v2_host_io_layout(plan: Plan) -> tuple[int, int, int]:
    """(in_bytes, out_bytes, io_bytes) of pa_v2_decode_host for `plan`."""
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    rc = lib().pa_v2_host_io_layout(ctypes.byref(plan.struct), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c))
    if rc != PA_OK:
        raise PaError(rc, "pa_v2_host_io_layout")
    return a.value, b.value, c.value


class HostStep:
    """pa_v2_decode_host with its buffers allocated once and its C arguments prepared once.

    pack(q, indices, indptr, last_page_len, first_page_offset) writes a step's host inputs into the pinned
    input buffer (or pass prepacked=True to run() after filling `host_in` yourself); run() makes the one
    C call and returns (out [B, Hq, D], lse2 [B, Hq]) as views of the pinned output buffer.
    graph_scale: also capture the step as a CUDA graph (pa_v2_host_graph_create) bound to this scale;
    run() with that scale then replays it (pa_v2_host_graph_run).
    mapped: the copy-free calls (pa_v2_decode_host_mapped / pa_v2_host_graph_create_mapped): the kernels
    read host_in and write host_out through their device mappings, and there is no device io buffer."""

    def __init__(self, plan: Plan, k_pool, v_pool, stream=None, graph_scale=None, mapped: bool = False):
        s = plan.struct
        self.plan = plan
        dev = k_pool.device
        self.in_bytes, self.out_bytes, self.io_bytes = pa_v2_host_io_layout(plan)
        self.host_in = torch.zeros(self.in_bytes, dtype=torch.uint8).pin_memory()
        self.host_out = torch.zeros(self.out_bytes, dtype=torch.uint8).pin_memory()
        self.mapped = bool(mapped)
        self.dev_io = None if mapped else torch.empty(self.io_bytes, dtype=torch.uint8, device=dev)
        ri, ti, oi = plan.device_arrays(dev)
        self.ws = (torch.empty(max(1, s.num_chunks), s.num_qo_heads, s.head_dim, device=dev),
                   torch.empty(max(1, s.num_chunks), s.num_qo_heads, device=dev))
        rows = s.batch * s.num_qo_heads
        self.words_in = self.host_in.view(torch.int32)
        self.q_words = rows * s.head_dim
        self.out = self.host_out[16:16 + rows * s.head_dim * 4].view(torch.float32).view(s.batch, s.num_qo_heads,
                                                                                           s.head_dim)
        self.lse = self.host_out[16 + rows * s.head_dim * 4:].view(torch.float32).view(s.batch, s.num_qo_heads)
        self._keep = (k_pool, v_pool, ri, ti, oi, stream)
        self._fn = lib().pa_v2_decode_host_mapped if mapped else lib().pa_v2_decode_host
        io = () if mapped else (self.dev_io.data_ptr(),)
        self._args = (ctypes.byref(s), self.host_in.data_ptr(), self.host_out.data_ptr(), *io,
                      _dev_ptr(k_pool, "k_pool"), _dev_ptr(v_pool, "v_pool"), KV_DTYPES[k_pool.dtype],
                      k_pool.shape[0], ri.data_ptr(), ti.data_ptr(), oi.data_ptr())
        self._tail = (self.ws[0].data_ptr(), self.ws[1].data_ptr(), _stream(stream))
        self._graph = None
        self._graph_scale = None
        if graph_scale is not None:
            g = ctypes.c_void_p()
            name = "pa_v2_host_graph_create_mapped" if mapped else "pa_v2_host_graph_create"
            rc = getattr(lib(), name)(*self._args, float(graph_scale), self.ws[0].data_ptr(), self.ws[1].data_ptr(),
                                      ctypes.byref(g))
            if rc != PA_OK:
                raise PaError(rc, name)
            self._graph, self._graph_scale = g, float(graph_scale)
            self._lib = lib()

    def __del__(self):
        if getattr(self, "_graph", None) is not None:
            self._lib.pa_v2_host_graph_destroy(self._graph)
            self._graph = None

    def pack(self, q, indices, indptr, last_page_len, first_page_offset):
        """Copy one step's inputs (host tensors) into the pinned input buffer."""
        w = self.words_in
        o = 0
        for t in (q.reshape(-1).view(torch.int32), indices, indptr, last_page_len, first_page_offset):
            n = t.numel()
            w[o:o + n] = t.reshape(-1).to(torch.int32)
            o += n
        w[o:] = 0

    def run(self, sm_scale: float):
        if self._graph is not None and float(sm_scale) == self._graph_scale:
            rc = self._lib.pa_v2_host_graph_run(self._graph, self._tail[2])
            if rc != PA_OK:
                raise PaError(rc, "pa_v2_host_graph_run")
            return self.out, self.lse
        rc = self._fn(*self._args, float(sm_scale), *self._tail)
        if rc != PA_OK:
            raise PaError(rc, "pa_v2_decode_host_mapped" if self.mapped else "pa_v2_decode_host")
        return self.out, self.lse


# ---------------------------------------------------------------------------
# second K stream (MLA / DSA)
# ---------------------------------------------------------------------------

def pa_v2_decode_partial_extra(plan: Plan, q, q_extra, k_pool, v_pool, k_extra_pool, indices, indptr,
                               last_page_len, first_page_offset, sm_scale: float, v_out=None, lse2_out=None,
                               status=None, stream=None, request_indices=None, kv_tile_indices=None):
    """Partial kernel with a second K stream (pa_v2_decode_partial_extra).

    Pools are device tensors [P, page_size, Hkv, width] whose last dimension is the row stride: k_pool and
    v_pool rows hold the 512-wide key / value part first (v_pool may be k_pool itself: MLA), k_extra_pool
    rows the 64-wide extra key.  Returns (v_out [N, Hq, 512], lse2_out [N, Hq])."""
    s = plan.struct
    dev = q.device
    if request_indices is None or kv_tile_indices is None:
        request_indices, kv_tile_indices, _ = plan.device_arrays(dev)
    if k_pool.dtype not in KV_DTYPES or v_pool.dtype != k_pool.dtype or k_extra_pool.dtype != k_pool.dtype:
        raise ValueError("k_pool, v_pool and k_extra_pool must share a 16-bit dtype")
    for name, t in (("k_pool", k_pool), ("v_pool", v_pool), ("k_extra_pool", k_extra_pool)):
        if t.dim() != 4 or tuple(t.shape[1:3]) != (s.page_size, s.num_kv_heads) or t.shape[0] != k_pool.shape[0]:
            raise ValueError(f"{name} must be [P, {s.page_size}, {s.num_kv_heads}, width]")
    if v_out is None:
        v_out = torch.empty(max(s.num_chunks, 1), s.num_qo_heads, s.head_dim, device=dev, dtype=torch.float32)
    if lse2_out is None:
        lse2_out = torch.empty(max(s.num_chunks, 1), s.num_qo_heads, device=dev, dtype=torch.float32)
    rc = lib().pa_v2_decode_partial_extra(
        ctypes.byref(s), _dev_ptr(q, "q", torch.float32), _dev_ptr(q_extra, "q_extra", torch.float32),
        _dev_ptr(k_pool, "k_pool"), k_pool.shape[3], _dev_ptr(v_pool, "v_pool"), v_pool.shape[3],
        _dev_ptr(k_extra_pool, "k_extra_pool"), k_extra_pool.shape[3], q_extra.shape[-1], KV_DTYPES[k_pool.dtype],
        k_pool.shape[0], _dev_ptr(indices, "indices", torch.int32), indices.numel(),
        _dev_ptr(indptr, "indptr", torch.int32), _dev_ptr(last_page_len, "last_page_len", torch.int32),
        _dev_ptr(first_page_offset, "first_page_offset", torch.int32),
        _dev_ptr(request_indices, "request_indices", torch.int32),
        _dev_ptr(kv_tile_indices, "kv_tile_indices", torch.int32), float(sm_scale),
        _dev_ptr(v_out, "v_out", torch.float32), _dev_ptr(lse2_out, "lse2_out", torch.float32),
        _dev_ptr(status, "status", torch.int32), _stream(stream))
    if rc != PA_OK:
        raise PaError(rc, "pa_v2_decode_partial_extra")
    return v_out, lse2_out


def decode_extra(plan: Plan, q, q_extra, k_pool, v_pool, k_extra_pool, indices, indptr, last_page_len,
                 first_page_offset, sm_scale: float, out=None, lse2=None, workspace=None, status=None, stream=None):
    """One second-K-stream decode step: pa_v2_decode_partial_extra, then pa_merge_states when the plan needs
    it.  Returns (out [B, Hq, 512], lse2 [B, Hq])."""
    s = plan.struct
    ri, ti, oi = plan.device_arrays(q.device)
    if not s.needs_merge:
        v, l = pa_v2_decode_partial_extra(plan, q, q_extra, k_pool, v_pool, k_extra_pool, indices, indptr,
                                          last_page_len, first_page_offset, sm_scale, out, lse2, status, stream,
                                          ri, ti)
        return v[:s.batch], l[:s.batch]
    wv, wl = workspace if workspace is not None else (None, None)
    wv, wl = pa_v2_decode_partial_extra(plan, q, q_extra, k_pool, v_pool, k_extra_pool, indices, indptr,
                                        last_page_len, first_page_offset, sm_scale, wv, wl, status, stream, ri, ti)
    return pa_merge_states(wv, wl, oi, s.batch, out, lse2, status, stream)



def pa_v2_selftest_wait(status, completed, limit_cycles: int, stream=None):
    """Bounded-wait self-test (pa_v2_selftest_wait): status int32 [1] and completed int32 [2], device tensors."""
    for name, t, n in (("status", status, 1), ("completed", completed, 2)):
        if not t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous() or t.numel() < n:
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor of >= {n} elements")
    rc = lib().pa_v2_selftest_wait(status.data_ptr(), completed.data_ptr(), int(limit_cycles), _stream(stream))
    if rc != PA_OK:
        raise PaError(rc, "pa_v2_selftest_wait")


def pa_v2_wave_fit_pages_per_chunk(indptr, ctas_per_chunk: int, wave: int) -> int:
    """Smallest pages_per_chunk whose CTA count fits one wave (pa_v2_wave_fit_pages_per_chunk); host indptr."""
    ip = torch.as_tensor(indptr, dtype=torch.int32).contiguous()
    v = int(lib().pa_v2_wave_fit_pages_per_chunk(ip.data_ptr(), ip.numel() - 1, int(ctas_per_chunk), int(wave)))
    if v <= 0:
        raise PaError(PA_EINVAL, "pa_v2_wave_fit_pages_per_chunk")
    return v


def pa_v2_balanced_pages_per_chunk(indptr, page_size: int, pages_per_chunk: int) -> int:
    """Largest pages_per_chunk <= the given one with its chunk count whose chunks give the tensor-core
    kernel's 8 warps equal stage counts, else the given one (pa_v2_balanced_pages_per_chunk); host indptr."""
    ip = torch.as_tensor(indptr, dtype=torch.int32).contiguous()
    v = int(lib().pa_v2_balanced_pages_per_chunk(ip.data_ptr(), ip.numel() - 1, int(page_size),
                                                 int(pages_per_chunk)))
    if v <= 0:
        raise PaError(PA_EINVAL, "pa_v2_balanced_pages_per_chunk")
    return v
