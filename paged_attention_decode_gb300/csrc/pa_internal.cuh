// pa_internal.cuh -- declarations shared by the partial-kernel translation units:
// the launch parameters, the chunk / stage geometry walked by every kernel
// variant, and the launchers each variant exports to the C-ABI entry point.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_device.cuh"
#include "pa_v2.h"

namespace pa {

constexpr int kWarps = 4;         // warps per CTA (each owns a private stage ring)
constexpr int kStageRows = 16;    // pool rows per stage
constexpr long long kWaitLimitCycles = 1ll << 31;  // bounded waits: ~1 s at 2 GHz

struct PartialParams {
  const float* q;
  const int32_t* indices;
  const int32_t* indptr;
  const int32_t* last_page_len;
  const int32_t* first_page_offset;
  const int32_t* request_indices;
  const int32_t* kv_tile_indices;
  const void* k_pool;   // used by the cp.async staging path
  const void* v_pool;
  float* v_out;        // partial workspace [num_chunks, Hq, D]
  float* lse_out;      // partial workspace [num_chunks, Hq]
  int32_t* status;
  // fused decode (pa_v2_decode): the last CTA of a (request, kv head, q-group)
  // merges that request's chunks into out / lse_final
  const int32_t* o_indptr;
  int32_t* counters;   // [batch * (CTA rows per chunk)], zero between launches
  float* out;          // [batch, Hq, D]
  float* lse_final;    // [batch, Hq]
  int32_t fused;
  // cascade level 0 (cascade-attention.md): M members' query heads stacked as one request,
  // h0 = kv * (M * Gm) + m * Gm + g; q and the final output stay in member layout [M, Hm, D]
  int32_t stack_members;   // M (1: no stacking)
  int32_t member_group;    // Gm = query heads per KV head of one member
  int32_t member_heads;    // Hm = query heads of one member
  int32_t out_row_step;    // final output row r is written at row r * out_row_step
  const int32_t* member_rows;  // stacked plans: request (q row group) of member m, or null for m
  const int32_t* out_rows;     // final output row of request r (member m when stacked), or null
  // partial rows (not fused): chunk c of request r (member m when stacked) goes to workspace row
  // part_rows[r] + c instead of row c, heads in member layout when stacked (one merge input holding
  // both cascade levels' chunks of each request, contiguously)
  const int32_t* part_rows;
  int64_t part_limit;          // rows x heads of the mapped workspace: a mapped row past it is skipped
  int64_t num_pages;
  int64_t num_indices;
  int32_t single_pages;  // > 0: a one-request plan of this many pages (chunk c is tile c of request 0)
  int32_t batch;
  int32_t num_qo_heads;
  int32_t num_kv_heads;
  int32_t group;       // Hq / Hkv
  int32_t hpc;         // query heads per CTA
  int32_t q_groups;
  int32_t page_size;
  int32_t pages_per_chunk;
  uint32_t ps_magic;   // fast division by page_size (see FastDiv)
  uint32_t ps_shift;
  float scale_log2;    // sm_scale * log2(e)
  int32_t warm_l2;     // prefetch each warp's first stage into L2 before waiting for the kernel before
};

// Division of a non-negative 32-bit n by a fixed divisor d >= 1 with one
// multiply-high, an add and a shift (Granlund & Montgomery, "Division by
// invariant integers using multiplication", 1994): with l = ceil(log2 d) and
// m = floor(2^32 * (2^l - d) / d) + 1, n / d = (mulhi(m, n) + n) >> l, exact
// for n < 2^31.
struct FastDiv {
  uint32_t magic, shift;
  static FastDiv make(uint32_t d) {
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    uint64_t m = ((1ull << 32) * ((1ull << l) - d)) / d + 1;
    return FastDiv{static_cast<uint32_t>(m), l};
  }
};

__device__ __forceinline__ uint32_t fast_div(uint32_t n, uint32_t magic, uint32_t shift) {
  return (__umulhi(magic, n) + n) >> shift;
}

// Row of q (in units of head_dim) that serves query head h of request r.
__device__ __forceinline__ size_t q_row(const PartialParams& p, int r, int h) {
  if (p.stack_members > 1) {
    const int within = h % p.group;  // position inside the KV head's stacked group
    const int m = within / p.member_group;
    const int hm = (h / p.group) * p.member_group + within % p.member_group;
    const int req = p.member_rows ? p.member_rows[m] : m;
    return (size_t)req * p.member_heads + hm;
  }
  return (size_t)r * p.num_qo_heads + h;
}

// Row of the final output / lse (in units of head_dim / 1) for query head h of request r.
__device__ __forceinline__ size_t out_row(const PartialParams& p, int r, int h) {
  if (p.stack_members > 1) {
    const int within = h % p.group;
    const int m = within / p.member_group;
    const int hm = (h / p.group) * p.member_group + within % p.member_group;
    const size_t row = p.out_rows ? (size_t)p.out_rows[m] : (size_t)m * p.out_row_step;
    return row * p.member_heads + hm;
  }
  const size_t row = p.out_rows ? (size_t)p.out_rows[r] : (size_t)r * p.out_row_step;
  return row * p.num_qo_heads + h;
}

// Workspace row (in units of head_dim) of chunk c's partial for query head h when the launch maps
// partial rows (p.part_rows): row part_rows[r] + c, or, stacked, part_rows[m] + c at member head hm.
// r: the chunk's request as validated by chunk_geom.
__device__ __forceinline__ size_t part_row(const PartialParams& p, int c, int r, int h) {
  if (p.stack_members > 1) {
    const int within = h % p.group;
    const int m = within / p.member_group;
    const int hm = (h / p.group) * p.member_group + within % p.member_group;
    return ((size_t)p.part_rows[m] + c) * p.member_heads + hm;
  }
  return ((size_t)p.part_rows[r] + c) * p.num_qo_heads + h;
}

struct ChunkGeom {
  int32_t slot_base;   // indptr[r]
  int32_t pages;       // pages of request r
  int32_t s_begin;     // first page slot of the chunk (relative to the request)
  int32_t s_end;       // one past the last slot
  int32_t fpo, lpl;
  int32_t n_stages;
  bool bad;            // request or page-slot range out of bounds (recorded in the status word)
};

struct StageGeom {
  int32_t slot;    // first page slot of the stage (relative to the request)
  int32_t npages;  // pages staged (small pages) or 1 (a 16-row slice of a large page)
  int32_t row0;    // first page row staged (slice offset for large pages)
  int32_t lo, hi;  // valid stage rows [lo, hi)
};

// Chunk c covers page slots [tile * ppc, min((tile + 1) * ppc, pages)) of its
// request; the kernel walks those slots directly.  A stage is 16 pool rows:
// floor(16 / ps) whole pages when ps <= 16, else one 16-row slice of a page.
//
// SPEC: a speculative read, made before the kernel has waited for the one
// before it, which may still be writing these arrays.  Loads go through L2 only
// (ld.global.cg: no L1 copy that could outlive the wait), every value is
// checked before it is used as an index, nothing is reported, and the result
// only ever chooses prefetch addresses (bad is set and n_stages is 0 when a
// value is out of range).
template <bool SPEC = false>
__device__ __forceinline__ ChunkGeom chunk_geom(const PartialParams& p, int c, int* r_out) {
  auto ld = [](const int32_t* a) -> int32_t { return SPEC ? __ldcg(a) : *a; };
  ChunkGeom g;
  int r = 0, tile = c;
  bool bad = false;
  if (p.single_pages > 0) {
    // one request: its page slots are 0 .. single_pages-1 (indptr = [0, num_indices] of the plan), and
    // chunk c is its tile c -- no chunk-array or indptr load stands before the first page-id load
    g.slot_base = 0;
    g.pages = p.single_pages;
  } else {
    r = ld(p.request_indices + c);
    tile = ld(p.kv_tile_indices + c);
    if (r < 0 || r >= p.batch) {
      if (!SPEC && threadIdx.x == 0) report(p.status, PA_DEVICE_BAD_REQUEST);
      bad = true;
      r = 0;
    }
    g.slot_base = ld(p.indptr + r);
    g.pages = ld(p.indptr + r + 1) - g.slot_base;
    if (!bad && (g.slot_base < 0 || g.pages < 0 || (int64_t)g.slot_base + g.pages > p.num_indices)) {
      if (!SPEC && threadIdx.x == 0) report(p.status, PA_DEVICE_BAD_SLOT);
      bad = true;
    }
    if (SPEC && (tile < 0 || (int64_t)tile * p.pages_per_chunk >= g.pages)) bad = true;
  }
  g.fpo = SPEC ? 0 : p.first_page_offset[r];
  g.lpl = SPEC ? p.page_size : p.last_page_len[r];
  g.s_begin = bad && SPEC ? 0 : tile * p.pages_per_chunk;
  g.s_end = min(g.s_begin + p.pages_per_chunk, g.pages);
  const int ps = p.page_size;
  if (bad || g.s_end <= g.s_begin) {
    g.n_stages = 0;
  } else if (ps <= kStageRows) {
    const int sp = kStageRows / ps;
    g.n_stages = (g.s_end - g.s_begin + sp - 1) / sp;
  } else {
    g.n_stages = (g.s_end - g.s_begin) * (ps / kStageRows);
  }
  g.bad = bad;
  *r_out = r;
  return g;
}

__device__ __forceinline__ StageGeom stage_geom(const ChunkGeom& g, int j, int ps) {
  StageGeom s;
  if (ps <= kStageRows) {
    const int sp = kStageRows / ps;
    s.slot = g.s_begin + j * sp;
    s.npages = min(sp, g.s_end - s.slot);
    s.row0 = 0;
    s.lo = (s.slot == 0) ? g.fpo : 0;
    s.hi = (s.slot + s.npages == g.pages) ? (s.npages - 1) * ps + g.lpl : s.npages * ps;
  } else {
    const int ns = ps / kStageRows;
    s.slot = g.s_begin + j / ns;
    s.npages = 1;
    s.row0 = (j % ns) * kStageRows;
    const int plo = (s.slot == 0) ? g.fpo : 0;
    const int phi = (s.slot == g.pages - 1) ? g.lpl : ps;
    s.lo = max(plo - s.row0, 0);
    s.hi = min(phi - s.row0, kStageRows);
  }
  return s;
}

// Merge the per-warp online-softmax states of a CTA of NW warps and write the
// chunk's normalized output and lse2: to workspace row `row` (a chunk), or,
// when final_output, to the final output of request `row`.  ms/ls:
// [NW][HP]; accs: [NW][HP] rows of DP >= D floats (unnormalized, relative to
// each warp's max).  Called by all threads after a __syncthreads() that
// follows the state writes.
//
// First one thread per head folds the warps' maxima into weights
// 2^(m_w - M) (kept in ms in place) and stores 1/L and the lse in ls[0][h] and
// ls[1][h]; then every thread combines float4 slices of the accumulators with
// those weights.  ms and ls are consumed.
// Query head h_first + h sits in state column h.
// MAPPED: partial rows follow p.part_rows (the cascade launch); other launches compile without it.
template <int HP, int D, int NW, bool MAPPED = false, int DP = D>
__device__ __forceinline__ void combine_warps_and_store(const PartialParams& p, float* ms, float* ls,
                                                        const float* accs, int row, int h_first, int nheads,
                                                        bool final_output, int req = 0) {
  static_assert(NW >= 2 && D % 4 == 0 && DP % 4 == 0, "float4 slices, two state rows for 1/L and lse");
  constexpr int Q = D / 4;  // float4 slices per head row
  const int tid = threadIdx.x;
  if (tid < nheads) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, ms[w * HP + tid]);
    float inv = 0.f, lse = -INFINITY;
    if (M != -INFINITY) {
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float wgt = fast_exp2(ms[w * HP + tid] - M);
        ms[w * HP + tid] = wgt;
        L += ls[w * HP + tid] * wgt;
      }
      inv = 1.f / L;
      lse = M + fast_log2(L);
    } else {
#pragma unroll
      for (int w = 0; w < NW; ++w) ms[w * HP + tid] = 0.f;
    }
    ls[tid] = inv;
    ls[HP + tid] = lse;
  }
  __syncthreads();
  for (int idx = tid; idx < nheads * Q; idx += NW * 32) {
    const int h = idx / Q;
    const int q = idx % Q;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float wgt = ms[w * HP + h];
      const float4 v = *reinterpret_cast<const float4*>(accs + (w * HP + h) * DP + 4 * q);
      a.x = fmaf(v.x, wgt, a.x);
      a.y = fmaf(v.y, wgt, a.y);
      a.z = fmaf(v.z, wgt, a.z);
      a.w = fmaf(v.w, wgt, a.w);
    }
    const float inv = ls[h];
    const float4 o = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
    size_t orow;
    float* dv;
    float* dl;
    if (final_output) {
      orow = out_row(p, row, h_first + h);
      dv = p.out;
      dl = p.lse_final;
    } else if (MAPPED) {
      orow = part_row(p, row, req, h_first + h);
      dv = p.v_out;
      dl = p.lse_out;
      if (orow >= (size_t)p.part_limit) {  // a row map pointing past the merge input: record, do not write
        report(p.status, PA_DEVICE_BAD_INDPTR);
        continue;
      }
    } else {
      orow = (size_t)row * p.num_qo_heads + h_first + h;
      dv = p.v_out;
      dl = p.lse_out;
    }
    reinterpret_cast<float4*>(dv + orow * D)[q] = o;
    if (q == 0) dl[orow] = ls[HP + h];
  }
}

// Fused merge (pa_v2_decode).  After a CTA has written its chunk's partial to
// the workspace, thread 0 takes a ticket on the counter of its (request, kv
// head, q-group) with an acq_rel atomic; the __syncthreads() before it makes
// the whole CTA's writes part of that release.  The CTA that takes the last
// ticket merges every chunk of the request for its heads with the closed form
// of issue #898, design piece 3 (m = max lse_i, w_i = 2^(lse_i - m),
// v = sum w_i v_i / sum w_i, lse = log2(sum w_i) + m) and resets the counter.
// No CTA waits on another: the first n-1 arrivals just leave.
//
// The merge is bound by L2 latency, so each thread issues all the loads of a
// batch at once: it owns one (head, 4-float slice) and a 1/split share of the
// chunks, reads up to 16 chunks' LSE and slice in one round, and folds them
// into a running (max, weight sum, accumulator) -- the same closed form applied
// batch by batch.  The shares of a slice then meet in shared memory.
// scratch: >= 6 * NW * 32 floats of shared memory no longer in use.
template <int D, int NW>
__device__ __forceinline__ void fused_merge(const PartialParams& p, float* scratch, int r, int h_first,
                                            int nheads, int num_chunks, int y, int ny) {
  __shared__ int s_last;
  constexpr int NT = NW * 32;
  constexpr int Q = D / 4;   // float4 slices per head row
  constexpr int B = 16;      // chunks per round of loads
  const int n0 = p.o_indptr[r];
  const int n1 = p.o_indptr[r + 1];
  if (n0 < 0 || n1 < n0 || n1 > num_chunks) {
    if (threadIdx.x == 0) report(p.status, PA_DEVICE_BAD_INDPTR);
    return;
  }
  __syncthreads();  // every thread's partial stores precede the release below
  if (threadIdx.x == 0) {
    int* ctr = p.counters + (size_t)r * ny + y;
    int prev;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(prev) : "l"(ctr) : "memory");
    const int last = prev == (n1 - n0) - 1;
    if (last) atomicExch(ctr, 0);  // every arrival is in: ready for the next launch
    s_last = last;
  }
  __syncthreads();
  if (!s_last) return;

  const int tid = threadIdx.x;
  const size_t hq = (size_t)p.num_qo_heads;
  const int units = nheads * Q;
  const int split = units >= NT ? 1 : NT / units;  // threads sharing one slice (chunk-parallel)
  const int sub = tid / units;
  float* sm_m = scratch;                                     // [NT]
  float* sm_w = scratch + NT;                                // [NT]
  float4* sm_a = reinterpret_cast<float4*>(scratch + 2 * NT);  // [NT]

  for (int ub = 0; ub < units; ub += NT) {
    const int u = ub + (tid % units);
    const bool working = sub < split && u < units;
    const int head = h_first + u / Q;
    const int quad = u % Q;
    float m = -INFINITY, W = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (working) {
      for (int c = n0 + sub; c < n1; c += B * split) {
        float l[B];
        float4 v[B];
#pragma unroll
        for (int k = 0; k < B; ++k) {
          const int cc = c + k * split;
          const bool ok = cc < n1;
          l[k] = ok ? __ldcg(p.lse_out + cc * hq + head) : -INFINITY;
          v[k] = ok ? __ldcg(reinterpret_cast<const float4*>(p.v_out + (cc * hq + head) * D) + quad)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float mb = m;
#pragma unroll
        for (int k = 0; k < B; ++k) mb = fmaxf(mb, l[k]);
        if (mb == -INFINITY) continue;
        const float sc = fast_exp2(m - mb);  // m = -inf -> 0
        W *= sc;
        acc.x *= sc;
        acc.y *= sc;
        acc.z *= sc;
        acc.w *= sc;
#pragma unroll
        for (int k = 0; k < B; ++k) {
          const float w = l[k] == -INFINITY ? 0.f : fast_exp2(l[k] - mb);
          W += w;
          acc.x = fmaf(w, v[k].x, acc.x);
          acc.y = fmaf(w, v[k].y, acc.y);
          acc.z = fmaf(w, v[k].z, acc.z);
          acc.w = fmaf(w, v[k].w, acc.w);
        }
        m = mb;
      }
    }
    if (split > 1) {
      sm_m[tid] = m;
      sm_w[tid] = W;
      sm_a[tid] = acc;
      __syncthreads();
      if (working && sub == 0) {
        float M = m;
        for (int s = 1; s < split; ++s) M = fmaxf(M, sm_m[tid + s * units]);
        float Wt = 0.f;
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
          for (int s = 0; s < split; ++s) {
            const int t2 = tid + s * units;
            const float sc = sm_m[t2] == -INFINITY ? 0.f : fast_exp2(sm_m[t2] - M);
            Wt += sm_w[t2] * sc;
            A.x += sm_a[t2].x * sc;
            A.y += sm_a[t2].y * sc;
            A.z += sm_a[t2].z * sc;
            A.w += sm_a[t2].w * sc;
          }
        }
        m = M;
        W = Wt;
        acc = A;
      }
    }
    if (working && sub == 0) {
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      float lse = -INFINITY;
      if (m != -INFINITY && W > 0.f) {
        o = make_float4(acc.x / W, acc.y / W, acc.z / W, acc.w / W);
        lse = m + fast_log2(W);
      }
      const size_t orow = out_row(p, r, head);
      reinterpret_cast<float4*>(p.out + orow * D)[quad] = o;
      if (quad == 0) p.lse_final[orow] = lse;
    }
  }
}

// The end of every partial kernel: write the chunk's state, then (fused
// decode) merge the request when this CTA is the last of its group.  A request
// with a single chunk writes straight to the final output.  scratch: the CTA's
// shared memory that is free once the states have been combined.
// num_chunks, y, ny: the launch's chunk count, this CTA's row among the CTAs of a chunk and their number
// (-1: the grid's own, gridDim.x, blockIdx.y, gridDim.y; a launch that runs two plans passes its plan's).
template <int HP, int D, int NW, bool MAPPED = false, int DP = D>
__device__ __forceinline__ void finish_chunk(const PartialParams& p, const ChunkGeom& g, float* ms,
                                             float* ls, const float* accs, float* scratch, int c, int r,
                                             int h_first, int nheads, int num_chunks = -1, int y = -1,
                                             int ny = -1) {
  if (MAPPED && g.bad) return;  // no row of a mapped workspace belongs to a chunk with a bad request
  bool direct = false;
  if (p.fused && !g.bad) {
    const int n0 = p.o_indptr[r], n1 = p.o_indptr[r + 1];
    direct = n1 - n0 == 1;
  }
  combine_warps_and_store<HP, D, NW, MAPPED, DP>(p, ms, ls, accs, direct ? r : c, h_first, nheads, direct, r);
  if (p.fused && !g.bad && !direct) {
    __syncthreads();  // scratch aliases the state arrays just read
    fused_merge<D, NW>(p, scratch, r, h_first, nheads, num_chunks < 0 ? (int)gridDim.x : num_chunks,
                       y < 0 ? (int)blockIdx.y : y, ny < 0 ? (int)gridDim.y : ny);
  }
}

// ---- launchers exported by the kernel translation units -------------------

struct LaunchArgs {
  PartialParams p;
  const CUtensorMap* tm_k;  // host copies, passed to the kernel by value
  const CUtensorMap* tm_v;
  int kv_dtype;
  int head_dim;
  int num_chunks;
  cudaStream_t stream;
};

// CUDA-core kernel (every dtype; the f32-pool path).  Returns PA_* status.
int launch_partial_simt(const LaunchArgs& a);
int occupancy_partial_simt(int kv_dtype, int head_dim, int hpc, int* blocks_per_sm);

// Tensor-core kernel (f16 / bf16 pools).  use_tma: stage with TMA (page sizes
// whose pages start on 8-row boundaries of a stage) instead of cp.async.
int launch_partial_tc(const LaunchArgs& a, bool use_tma);
// Two plans over the same pools in one launch: a's plan on CTA columns [0, a.num_chunks), p1's n1 chunks
// after them (the cascade levels); both plans fused (each CTA group merges its own requests).
int launch_partial_tc_two_plans(const LaunchArgs& a, const PartialParams& p1, int n1, bool use_tma);
int occupancy_partial_tc(int kv_dtype, int head_dim, int hpc, bool use_tma, int* blocks_per_sm);

// Second-K-stream kernels (head_dim 512 + extra 64; f16 / bf16 pools): CUDA
// cores (pa_partial_extra.cu) and tensor cores (pa_partial_extra_tc.cu).
int occupancy_partial_extra(int kv_dtype, int* blocks_per_sm);
int occupancy_partial_extra_tc(int kv_dtype, int* blocks_per_sm);
int launch_partial_extra_tc(const PartialParams& p, const void* q_extra, const void* k_extra, int64_t k_stride,
                            int64_t v_stride, int64_t e_stride, bool shared_v, int kv_dtype, dim3 grid,
                            cudaStream_t stream);
// The tensor-memory (tcgen05) second-K-stream kernel: values read from the key
// tile, up to 32 query heads per CTA (p.hpc <= 32).
int occupancy_partial_extra_tc05(int kv_dtype, int* blocks_per_sm);
int launch_partial_extra_tc05(const PartialParams& p, const void* q_extra, const void* k_extra, int64_t k_stride,
                              int64_t e_stride, int kv_dtype, dim3 grid, cudaStream_t stream);

// True when the tensor-core kernel stages this page size with TMA.
inline bool tc_uses_tma(int page_size) {
  return page_size % 8 == 0 && (page_size <= kStageRows || page_size % kStageRows == 0);
}

// Launch `fn` as a programmatic dependent of the kernel before it in the
// stream: its CTAs may become resident while that kernel is finishing, and
// each one waits (griddepcontrol.wait) for it to complete before its first
// global-memory access.  Without a programmatic predecessor the wait is a no-op.
template <typename... Params, typename... Args>
inline cudaError_t launch_dependent(void (*fn)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                    Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, static_cast<Args&&>(args)...);
}

// Shared-memory opt-in above 48 KB, once per kernel and device (safe to call
// under stream capture after the first call).
bool prepare_kernel(const void* fn, size_t smem);

}  // namespace pa
