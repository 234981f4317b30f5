// pa_partial_extra_tc.cu -- tensor-core variant of the second-K-stream partial
// kernel (MLA / DSA decode).
//
// Same contract as the CUDA-core variant in pa_partial_extra.cu
// (sparse-paged-decode.md, issue #904, the DSA paragraphs, third way out):
//   score_t = scale * (q . k[row_t][0:512]) + scale * (q_extra . k_extra[row_t][0:64]),
// output = softmax-weighted sum of v[row_t][0:512], rows resolved through the
// CSR page table, one CTA per (chunk, kv head, group of 8 query heads).
//
// Structure (the one the single-stream tensor-core kernel uses): 8 warps (4 when
// values have their own allocation), each staging its own 16-row stages with
// cp.async 16-byte copies into 128-byte-swizzled half rows; per stage and warp
//   S^T [16 tokens x 8 heads] = K [16 x 576] . Q^T [576 x 8]     (tokens are M)
//   O^T [512 x 8 heads]      += V^T [512 x 16] . P^T [16 x 8]
// with warp-level mma.sync m16n8k16 (f32 accumulate).  Q (hi + lo halves of
// the pool's 16-bit type, scale * log2(e) folded in) sits once per CTA in a
// swizzled shared tile and enters every k-step through ldmatrix; the online
// softmax lives in the MMA C-fragment layout; P^T goes through a per-warp
// shared transpose; O^T (128 f32 registers per thread) stays in registers for
// the whole chunk.  When v_pool is k_pool (MLA) the values are read from the
// key tile.  At the end the warps' states merge through shared memory.
// Inside the stage loop there is no block barrier: warps synchronise only
// with themselves.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "pa_internal.cuh"
#include "pa_mma.cuh"

namespace pa {
namespace {

constexpr int kMDim = 512;                 // Dim (key part and value width)
constexpr int kMExtra = 64;                // ExtraDim
constexpr int kMHeads = 8;                 // query heads per CTA: one n-tile
constexpr int kMKSteps = (kMDim + kMExtra) / 16;   // 36 k-steps of S^T
constexpr int kMDimSteps = kMDim / 16;             // 32 (the latent part; also the O^T m-tiles)
constexpr int kMChunksK = kMDim / 8;               // 64 16-byte chunks per latent row
constexpr int kMChunksE = kMExtra / 8;             // 8 per extra row
constexpr int kMQRow = (kMDim + kMExtra) * 2;      // bytes of one head's q row in shared memory

// NW warps per CTA, each with NSW stages in flight.
template <bool SHARED_V, int NW, int NSW_>
struct MlaLayout {
  static constexpr int kMWarps = NW;
  static constexpr int NSW = NSW_;
  static constexpr int KT = (kMDim / 64) * 2048;              // 16 rows x 512: 8 half-tiles of 2 KB
  static constexpr int ET = (kMExtra / 64) * 2048;            // 16 rows x 64
  static constexpr int STAGE = KT + ET + (SHARED_V ? 0 : KT);
  static constexpr int RING = kMWarps * NSW * STAGE;
  static constexpr int STATE = kMWarps * kMHeads * kMDim * 4;  // per-warp O^T for the final merge
  static constexpr int BODY = RING > STATE ? RING : STATE;
  static constexpr int QHALF = kMHeads * kMQRow;               // 9216: q hi, then q lo
  static constexpr int QOFF = BODY;
  static constexpr int PTOFF = QOFF + 2 * QHALF;              // per warp P^T hi/lo [8 heads][16 tokens]
  static constexpr int MSOFF = PTOFF + kMWarps * 2 * kMHeads * 16 * 2;
  static constexpr int TOTAL = MSOFF + 2 * kMWarps * kMHeads * 4;
  static constexpr int ALLOC = TOTAL + 128;
};

struct ExtraTcFields {
  const float* q_extra;
  const void* k_extra;
  int64_t k_stride, v_stride, e_stride;
};

// Byte offset of 16-byte chunk `ch` (0 .. 71) of head row `h` (0 .. 7) in the
// q tile: rows of 1152 bytes, chunk index XOR h within each group of 8, so the
// 8 rows of an ldmatrix phase fall in 8 distinct bank groups.
__device__ __forceinline__ uint32_t qswz(int h, int ch) { return (uint32_t)(h * kMQRow + ((ch ^ h) << 4)); }

// Registers capped at 224 (no spills): the O^T tile alone takes 128 per thread.
template <typename T, bool SHARED_V, int NW, int NSW_>
__global__ void __maxnreg__(224)
    pa_v2_partial_extra_tc_kernel(const PartialParams p, const ExtraTcFields x) {
  using L = MlaLayout<SHARED_V, NW, NSW_>;
  constexpr int NSW = L::NSW;
  constexpr int kMWarps = NW;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
  float* accs = reinterpret_cast<float*>(smem);
  float* ms = reinterpret_cast<float*>(smem + L::MSOFF);
  float* ls = ms + kMWarps * kMHeads;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  const int c = blockIdx.x;
  const int kvh = blockIdx.y / p.q_groups;
  const int qg = blockIdx.y % p.q_groups;
  const int h_first = kvh * p.group + qg * p.hpc;
  const int nheads = min(p.hpc, p.group - qg * p.hpc);
  const int ps = p.page_size;

  pdl_launch_dependents();
  pdl_wait_prerequisites();

  int r;
  const ChunkGeom gm = chunk_geom(p, c, &r);
  unsigned char* mst = smem + warp * NSW * L::STAGE;
  unsigned short* pt_hi = reinterpret_cast<unsigned short*>(smem + L::PTOFF) + warp * 2 * kMHeads * 16;
  unsigned short* pt_lo = pt_hi + kMHeads * 16;
  const uint64_t policy = policy_evict_first();
  const T* kpool = static_cast<const T*>(p.k_pool);
  const T* vpool = static_cast<const T*>(p.v_pool);
  const T* epool = static_cast<const T*>(x.k_extra);

  // Lane (lane & 15) holds the page id of page (lane & 15) of stage j, or -1.
  auto stage_page = [&](int j) -> int32_t {
    if (j >= gm.n_stages) return -1;
    const StageGeom s = stage_geom(gm, j, ps);
    const int tp = lane & 15;
    if (tp >= s.npages) return -1;
    return __ldg(p.indices + gm.slot_base + s.slot + tp);
  };

  // Stage j of this warp into ring slot `slot`.  Lane l copies row l & 15 of the
  // stage, chunks (l >> 4) + 2k of its latent [and value] and extra parts: the
  // row's page is resolved once per stage.
  auto issue = [&](int j, int slot, int32_t my_page) {
    const StageGeom s = stage_geom(gm, j, ps);
    const int nrows = ps <= kStageRows ? s.npages * ps : kStageRows;
    const uint32_t kdst = smem_addr(mst + slot * L::STAGE);
    const uint32_t edst = kdst + L::KT;
    const uint32_t vdst = edst + L::ET;
    const int row = lane & 15;
    const int half = lane >> 4;
    const int sl = ps <= kStageRows ? (int)fast_div((uint32_t)row, p.ps_magic, p.ps_shift) : 0;
    const int e = ps <= kStageRows ? row - sl * ps : s.row0 + row;
    const int32_t page = __shfl_sync(0xffffffffu, my_page, sl & 15);
    if (row < nrows) {
      if (page >= 0 && (int64_t)page < p.num_pages) {
        const int64_t prow = ((int64_t)page * ps + e) * p.num_kv_heads + kvh;
        const T* ksrc = kpool + prow * x.k_stride;
        const T* vsrc = vpool + prow * x.v_stride;
#pragma unroll 8
        for (int k = 0; k < kMChunksK / 2; ++k) {
          const int ch = half + 2 * k;
          cp_async_16(kdst + swz(row, ch), ksrc + ch * 8, policy);
          if (!SHARED_V) cp_async_16(vdst + swz(row, ch), vsrc + ch * 8, policy);
        }
        const T* esrc = epool + prow * x.e_stride;
#pragma unroll
        for (int k = 0; k < kMChunksE / 2; ++k) {
          const int ch = half + 2 * k;
          cp_async_16(edst + swz(row, ch), esrc + ch * 8, policy);
        }
      } else if (half == 0) {
        report(p.status, PA_DEVICE_BAD_PAGE);
      }
    }
  };

#pragma unroll
  for (int s = 0; s < NSW; ++s) {
    const int j = warp + s * kMWarps;
    if (j < gm.n_stages) issue(j, s, stage_page(j));
    cp_async_commit();
  }
  int32_t next_page = stage_page(warp + NSW * kMWarps);

  // ---- Q^T tile (hi + lo halves) in shared memory, once per CTA ----
  {
    // a thread's q loads are issued 12 at a time before its shared-memory stores, so they
    // overlap instead of paying one memory latency each
    unsigned char* qhi = smem + L::QOFF;
    unsigned char* qlo = qhi + L::QHALF;
    constexpr int kTotal = kMHeads * (kMDim + kMExtra);
    constexpr int kBatch = 12;
#pragma unroll 1
    for (int base = 0; base < kTotal; base += kBatch * kMWarps * 32) {
      float qv[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int idx = base + threadIdx.x + k * kMWarps * 32;
        const int h = idx / (kMDim + kMExtra);
        const int d = idx - h * (kMDim + kMExtra);
        qv[k] = 0.f;
        if (idx < kTotal && h < nheads) {
          const size_t qrow = (size_t)r * p.num_qo_heads + h_first + h;
          qv[k] = d < kMDim ? __ldg(p.q + qrow * kMDim + d) : __ldg(x.q_extra + qrow * kMExtra + (d - kMDim));
        }
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int idx = base + threadIdx.x + k * kMWarps * 32;
        if (idx < kTotal) {
          const int h = idx / (kMDim + kMExtra);
          const int d = idx - h * (kMDim + kMExtra);
          const float v = qv[k] * p.scale_log2;
          const float hi = TC<T>::round(v);
          const uint32_t off = qswz(h, d >> 3) + (d & 7) * 2;
          *reinterpret_cast<unsigned short*>(qhi + off) = TC<T>::bits(hi);
          *reinterpret_cast<unsigned short*>(qlo + off) = TC<T>::bits(v - hi);
        }
      }
    }
  }
  __syncwarp();     // reconverge the per-thread branches before the aligned barrier
  __syncthreads();  // the q tile is complete (the only block barrier before the end of the chunk)
  const uint32_t qbase = smem_addr(smem + L::QOFF);

  float o[kMDimSteps][4];
#pragma unroll
  for (int mt = 0; mt < kMDimSteps; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[mt][e] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

  const int krow = ((lane >> 3) & 1) * 8 + (lane & 7);  // K fragment row this lane addresses
  const int vtok = (lane >> 4) * 8 + (lane & 7);        // V^T fragment token this lane addresses
  const int qrow_l = lane & 7;                          // q tile row (head) this lane addresses
  const uint32_t qhalf_l = (lane >> 4) ? (uint32_t)L::QHALF : 0u;
  const int qchunk_l = (lane >> 3) & 1;

  int i = 0;
  for (;; ++i) {
    const int j = warp + i * kMWarps;
    if (j >= gm.n_stages) break;
    const int slot = i % NSW;
    cp_async_wait<NSW - 1>();
    __syncwarp();
    const StageGeom sg = stage_geom(gm, j, ps);
    unsigned char* kt = mst + slot * L::STAGE;
    unsigned char* vt = SHARED_V ? kt : kt + L::KT + L::ET;
    const uint32_t kbase = smem_addr(kt);
    const uint32_t ebase = kbase + L::KT;
    const uint32_t vbase = smem_addr(vt);

    // rows of the value tile outside [lo, hi) may hold stale or non-finite data: zero them
    if (sg.lo > 0 || sg.hi < kStageRows) {
      for (int idx = lane; idx < kStageRows * kMChunksK; idx += 32) {
        const int row = idx / kMChunksK;
        if (row < sg.lo || row >= sg.hi)
          *reinterpret_cast<uint4*>(vt + swz(row, idx % kMChunksK)) = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
    }

    // ---- S^T = K . Q^T: hi and lo halves, even and odd k-steps in separate accumulators ----
    float sacc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[a][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < kMKSteps; ++ks) {
      uint32_t a[4], b[4];
      if (ks < kMDimSteps) ldsm_x4(a, kbase + swz(krow, ks * 2 + (lane >> 4)));
      else ldsm_x4(a, ebase + swz(krow, (ks - kMDimSteps) * 2 + (lane >> 4)));
      ldsm_x4(b, qbase + qhalf_l + qswz(qrow_l, ks * 2 + qchunk_l));  // hi b0 b1, lo b0 b1
      TC<T>::mma(sacc[ks & 1], a, b[0], b[1]);
      TC<T>::mma(sacc[2 + (ks & 1)], a, b[2], b[3]);
    }

    // ---- online softmax over the stage (tokens g and g + 8, heads 2t, 2t + 1) ----
    const bool v0 = g >= sg.lo && g < sg.hi;
    const bool v1 = g + 8 >= sg.lo && g + 8 < sg.hi;
    float sv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) sv[e] = (sacc[0][e] + sacc[1][e]) + (sacc[2][e] + sacc[3][e]);
    const float s0 = v0 ? sv[0] : -INFINITY;
    const float s1 = v0 ? sv[1] : -INFINITY;
    const float s2 = v1 ? sv[2] : -INFINITY;
    const float s3 = v1 ? sv[3] : -INFINITY;
    float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
    const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
    const float a0 = fast_exp2(m_run[0] - mu0), a1 = fast_exp2(m_run[1] - mu1);
    m_run[0] = mn0;
    m_run[1] = mn1;
    float pr[4];
    pr[0] = fast_exp2(s0 - mu0);
    pr[1] = fast_exp2(s1 - mu1);
    pr[2] = fast_exp2(s2 - mu0);
    pr[3] = fast_exp2(s3 - mu1);
    l_run[0] = l_run[0] * a0 + pr[0] + pr[2];
    l_run[1] = l_run[1] * a1 + pr[1] + pr[3];
#pragma unroll
    for (int mt = 0; mt < kMDimSteps; ++mt) {
      o[mt][0] *= a0;
      o[mt][1] *= a1;
      o[mt][2] *= a0;
      o[mt][3] *= a1;
    }
    // P^T [head][token] for the B operand, hi and lo
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int hh = 2 * t + (e & 1);
      const int tok = g + (e >> 1) * 8;
      const float hi = TC<T>::round(pr[e]);
      pt_hi[hh * 16 + tok] = TC<T>::bits(hi);
      pt_lo[hh * 16 + tok] = TC<T>::bits(pr[e] - hi);
    }
    __syncwarp();

    // ---- O^T += V^T . P^T ----
    uint32_t bp[4];
    {
      const unsigned short* src = (lane >> 4) ? pt_lo : pt_hi;
      ldsm_x4(bp, smem_addr(src + (lane & 7) * 16 + ((lane >> 3) & 1) * 8));
    }
#pragma unroll
    for (int mt = 0; mt < kMDimSteps; ++mt) {
      uint32_t a[4];
      ldsm_x4_trans(a, vbase + swz(vtok, mt * 2 + ((lane >> 3) & 1)));
      TC<T>::mma(o[mt], a, bp[0], bp[1]);
      TC<T>::mma(o[mt], a, bp[2], bp[3]);
    }
    __syncwarp();  // every lane's reads of the slot and of P^T are done

    // refill this slot with the warp's stage NSW rounds ahead
    const int jn = warp + (i + NSW) * kMWarps;
    if (jn < gm.n_stages) {
      issue(jn, slot, next_page);
      next_page = stage_page(jn + kMWarps);
    }
    cp_async_commit();
    __syncwarp();
  }
  cp_async_wait<0>();

  // ---- per-warp state -> shared memory, then merge the warps ----
#pragma unroll
  for (int e = 0; e < 2; ++e)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) l_run[e] += __shfl_xor_sync(0xffffffffu, l_run[e], off);
  __syncthreads();  // all warps are done with their stages: reuse them for the states
#pragma unroll
  for (int mt = 0; mt < kMDimSteps; ++mt) {
    float* a0 = accs + (warp * kMHeads + 2 * t) * kMDim + 16 * mt + g;
    float* a1 = a0 + kMDim;
    a0[0] = o[mt][0];
    a1[0] = o[mt][1];
    a0[8] = o[mt][2];
    a1[8] = o[mt][3];
  }
  if (g == 0) {
    ms[warp * kMHeads + 2 * t] = m_run[0];
    ms[warp * kMHeads + 2 * t + 1] = m_run[1];
    ls[warp * kMHeads + 2 * t] = l_run[0];
    ls[warp * kMHeads + 2 * t + 1] = l_run[1];
  }
  __syncwarp();
  __syncthreads();
  combine_warps_and_store<kMHeads, kMDim, kMWarps>(p, ms, ls, accs, c, h_first, nheads, false);
}

}  // namespace

using ExtraTcKernel = void (*)(const PartialParams, const ExtraTcFields);

namespace {

// Values in the key tile (MLA): 8 warps with one stage each (measured faster
// on GB300 than 4 warps with two: 156 vs 219 us for 16 DSA requests); separate
// values (twice the stage bytes): 4 warps, one stage each.
constexpr int kMlaWarps = 8;
constexpr int kMlaRing = 1;
using SharedL = MlaLayout<true, kMlaWarps, kMlaRing>;
using SeparateL = MlaLayout<false, 4, 1>;

int extra_tc_warps(bool shared_v) { return shared_v ? kMlaWarps : 4; }

ExtraTcKernel extra_tc_pick(int kv_dtype, bool shared_v, size_t* smem) {
  *smem = shared_v ? SharedL::ALLOC : SeparateL::ALLOC;
  if (kv_dtype == PA_F16)
    return shared_v ? pa_v2_partial_extra_tc_kernel<__half, true, kMlaWarps, kMlaRing>
                    : pa_v2_partial_extra_tc_kernel<__half, false, 4, 1>;
  if (kv_dtype == PA_BF16)
    return shared_v ? pa_v2_partial_extra_tc_kernel<__nv_bfloat16, true, kMlaWarps, kMlaRing>
                    : pa_v2_partial_extra_tc_kernel<__nv_bfloat16, false, 4, 1>;
  return nullptr;
}

}  // namespace

int occupancy_partial_extra_tc(int kv_dtype, int* blocks_per_sm) {
  size_t smem = 0;
  ExtraTcKernel fn = extra_tc_pick(kv_dtype, true, &smem);
  if (!fn) return PA_EUNSUPPORTED;
  if (!prepare_kernel(reinterpret_cast<const void*>(fn), smem)) return PA_ECUDA;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, extra_tc_warps(true) * 32, smem) ==
                 cudaSuccess
             ? PA_OK
             : PA_ECUDA;
}

int launch_partial_extra_tc(const PartialParams& p, const void* q_extra, const void* k_extra, int64_t k_stride,
                            int64_t v_stride, int64_t e_stride, bool shared_v, int kv_dtype, dim3 grid,
                            cudaStream_t stream) {
  size_t smem = 0;
  ExtraTcKernel fn = extra_tc_pick(kv_dtype, shared_v, &smem);
  if (!fn) return PA_EUNSUPPORTED;
  if (!prepare_kernel(reinterpret_cast<const void*>(fn), smem)) return PA_ECUDA;
  ExtraTcFields x;
  x.q_extra = static_cast<const float*>(q_extra);
  x.k_extra = k_extra;
  x.k_stride = k_stride;
  x.v_stride = v_stride;
  x.e_stride = e_stride;
  const cudaError_t rc = launch_dependent(fn, grid, dim3(extra_tc_warps(shared_v) * 32), smem, stream, p, x);
  return rc == cudaSuccess && cudaGetLastError() == cudaSuccess ? PA_OK : PA_ECUDA;
}

}  // namespace pa
