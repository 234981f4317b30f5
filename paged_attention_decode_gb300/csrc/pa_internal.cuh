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
  float* v_out;
  float* lse_out;
  int32_t* status;
  int64_t num_pages;
  int64_t num_indices;
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

struct ChunkGeom {
  int32_t slot_base;   // indptr[r]
  int32_t pages;       // pages of request r
  int32_t s_begin;     // first page slot of the chunk (relative to the request)
  int32_t s_end;       // one past the last slot
  int32_t fpo, lpl;
  int32_t n_stages;
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
__device__ __forceinline__ ChunkGeom chunk_geom(const PartialParams& p, int c, int* r_out) {
  ChunkGeom g;
  int r = p.request_indices[c];
  const int tile = p.kv_tile_indices[c];
  bool bad = false;
  if (r < 0 || r >= p.batch) {
    if (threadIdx.x == 0) report(p.status, PA_DEVICE_BAD_REQUEST);
    bad = true;
    r = 0;
  }
  g.slot_base = p.indptr[r];
  g.pages = p.indptr[r + 1] - g.slot_base;
  if (!bad && (g.slot_base < 0 || g.pages < 0 || (int64_t)g.slot_base + g.pages > p.num_indices)) {
    if (threadIdx.x == 0) report(p.status, PA_DEVICE_BAD_SLOT);
    bad = true;
  }
  g.fpo = p.first_page_offset[r];
  g.lpl = p.last_page_len[r];
  g.s_begin = tile * p.pages_per_chunk;
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

// Merge the per-warp online-softmax states of a CTA and write the chunk's
// normalized output and lse2.  ms/ls: [kWarps][HP]; accs: [kWarps][HP][D]
// (unnormalized, relative to each warp's max).  Called by all threads after a
// __syncthreads() that follows the state writes.
template <int HP, int D>
__device__ __forceinline__ void combine_warps_and_store(const PartialParams& p, const float* ms, const float* ls,
                                                        const float* accs, int c, int h_first, int nheads) {
  for (int idx = threadIdx.x; idx < nheads * D; idx += kWarps * 32) {
    const int h = idx / D;
    const int d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ms[w * HP + h]);
    float out = 0.f, lse = -INFINITY;
    if (M != -INFINITY) {
      float L = 0.f, A = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float wgt = fast_exp2(ms[w * HP + h] - M);
        L += ls[w * HP + h] * wgt;
        A += accs[(w * HP + h) * D + d] * wgt;
      }
      out = A / L;
      lse = M + fast_log2(L);
    }
    const size_t row = (size_t)c * p.num_qo_heads + h_first + h;
    p.v_out[row * D + d] = out;
    if (d == 0) p.lse_out[row] = lse;
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
int occupancy_partial_tc(int kv_dtype, int head_dim, int hpc, bool use_tma, int* blocks_per_sm);

// True when the tensor-core kernel stages this page size with TMA.
inline bool tc_uses_tma(int page_size) {
  return page_size % 8 == 0 && (page_size <= kStageRows || page_size % kStageRows == 0);
}

// Shared-memory opt-in above 48 KB, once per kernel and device (safe to call
// under stream capture after the first call).
bool prepare_kernel(const void* fn, size_t smem);

}  // namespace pa
