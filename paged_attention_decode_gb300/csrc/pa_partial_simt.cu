// pa_partial_simt.cu -- CUDA-core variant of the split-KV partial kernel.
//
// What it computes (issue #898 "Fused paged-attention decode v2: CSR page
// table, cross-CTA split-KV, and variable-length merge kernels", design pieces
// 1-2 and Task 2; PR #984 "fused paged-attention decode v2 with CSR page table
// and cross-CTA split-KV", What changed 2): one CTA owns one (chunk, kv head,
// q-head group) triple, walks the chunk's pages through the CSR page table,
// reads every K/V element of that KV head once and reuses it for all query
// heads of the group, runs an online softmax in base 2 (log2(e) folded into
// the scale) in f32, and writes the chunk's normalized output and its log2-LSE.
//
// This variant serves f32 pools (and any dtype on request).  Mapping:
//  - K/V staging: each of the CTA's 4 warps owns a private ring of stages in
//    shared memory, filled by TMA (cp.async.bulk.tensor, 3-D tensor map over
//    the pool viewed as [pool rows, Hkv, D]) and completed on an mbarrier.
//    Warps take stages round-robin.
//  - Scores: a K row is split over LPT lanes (16 bytes each: 128-bit shared
//    loads); the per-head partial dot products are reduce-scattered across
//    those lanes with warp shuffles so each lane ends up owning one head's
//    score.  Softmax state is rescaled once per 16-row stage.
//  - Output: per-warp states are merged through shared memory at the end of
//    the chunk and written as a normalized partial plus lse2.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "pa_internal.cuh"

namespace pa {
namespace {

// ---- K/V element loading: 16 bytes of one row -> VEC floats ---------------

template <typename T> struct KV;

template <> struct KV<float> {
  static constexpr int VEC = 4;
  __device__ __forceinline__ static void load(const float* p, float (&f)[4]) {
    float4 v = *reinterpret_cast<const float4*>(p);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
};

template <> struct KV<__half> {
  static constexpr int VEC = 8;
  __device__ __forceinline__ static void load(const __half* p, float (&f)[8]) {
    uint4 raw = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
};

template <> struct KV<__nv_bfloat16> {
  static constexpr int VEC = 8;
  // bfloat16 is the upper half of a binary32: widening is a shift / mask.
  __device__ __forceinline__ static void load(const __nv_bfloat16* p, float (&f)[8]) {
    uint4 raw = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};

// Sum HP per-lane partial dot products over the LPT lanes that share a row
// (lanes differ in the low bits `dl`).  At each butterfly level where more
// than one head remains, a lane keeps the half of the heads selected by its
// `dl` bit and sends the other half, so the head set halves per level; the
// remaining levels are a plain butterfly sum.  Afterwards lanes
// [h * LPT/HP, (h+1) * LPT/HP) of the row hold the full score of head h.
// Shuffles per row group: (HP - 1) + log2(LPT / HP).
template <int HP, int LPT>
__device__ __forceinline__ float reduce_scatter(float (&part)[HP], int dl) {
  constexpr int LEVELS = LPT == 32 ? 5 : LPT == 16 ? 4 : LPT == 8 ? 3 : LPT == 4 ? 2 : LPT == 2 ? 1 : 0;
#pragma unroll
  for (int lvl = 0; lvl < LEVELS; ++lvl) {
    const int o = LPT >> (lvl + 1);
    const int cnt = HP >> lvl;  // heads still held per lane
    if (cnt > 1) {
      const bool upper = (dl & o) != 0;
#pragma unroll
      for (int h = 0; h < HP / 2; ++h) {
        if (h < cnt / 2) {
          const float send = upper ? part[h] : part[h + cnt / 2];
          const float keep = upper ? part[h + cnt / 2] : part[h];
          part[h] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
    } else {
      part[0] += __shfl_xor_sync(0xffffffffu, part[0], o);
    }
  }
  return part[0];
}

// ---- the kernel -------------------------------------------------------------

// T: pool element type.  D: head dim.  HP: query heads per CTA, padded to a
// power of two.  NSW: ring depth per warp.
template <typename T, int D, int HP, int NSW>
__global__ void __launch_bounds__(kWarps * 32)
    pa_v2_partial_simt_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const PartialParams p) {
  constexpr int VEC = KV<T>::VEC;
  constexpr int LPT = D / VEC;          // lanes per K/V row
  constexpr int TPW = 32 / LPT;         // rows per warp step
  constexpr int NSTEP = kStageRows / TPW;
  static_assert(HP <= LPT, "reduce-scatter needs at least one lane per head");
  constexpr int LPH = LPT / HP;         // lanes holding each head's score
  constexpr int SIDE = kStageRows * D;  // elements per side per stage

  constexpr size_t STAGE_BYTES = sizeof(T) * kWarps * NSW * 2 * SIDE;
  constexpr size_t STATE_BYTES = sizeof(float) * kWarps * HP * D;
  constexpr size_t BODY_BYTES = STAGE_BYTES > STATE_BYTES ? STAGE_BYTES : STATE_BYTES;

  extern __shared__ __align__(128) unsigned char smem[];
  T* stages = reinterpret_cast<T*>(smem);                          // [kWarps][NSW][2][kStageRows][D]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BODY_BYTES);  // [kWarps][NSW]
  float* ms = reinterpret_cast<float*>(bars + kWarps * NSW);  // [kWarps][HP]
  float* ls = ms + kWarps * HP;                                  // [kWarps][HP]
  float* accs = reinterpret_cast<float*>(smem);                 // [kWarps][HP][D], reuses the stages

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tl = lane / LPT;  // row of the warp step this lane reads
  const int dl = lane % LPT;  // 16-byte slice of the row
  const int hs = dl / LPH;    // head whose score this lane owns after the reduction
  const int c = blockIdx.x;
  const int kvh = blockIdx.y / p.q_groups;
  const int qg = blockIdx.y % p.q_groups;
  const int h_first = kvh * p.group + qg * p.hpc;
  const int nheads = min(p.hpc, p.group - qg * p.hpc);
  const int ps = p.page_size;

  // the kernel that follows (the merge, or the next step) may be scheduled now;
  // it waits for this grid to finish
  pdl_launch_dependents();

  // launched as a programmatic dependent: the kernel before this one in the
  // stream has completed, and its writes are visible, once this returns
  pdl_wait_prerequisites();

  // ---- chunk geometry ----
  int r;
  const ChunkGeom g = chunk_geom(p, c, &r);

  // ---- barriers ----
  uint64_t* mybar = bars + warp * NSW;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NSW; ++s) mbar_init(&mybar[s], 1);
    fence_barrier_init();
  }
  __syncwarp();


  T* mystages = stages + (size_t)warp * NSW * 2 * SIDE;
  const uint64_t policy = policy_evict_first();
  const int box_rows = ps <= kStageRows ? ps : kStageRows;

  // Page id this lane needs to issue stage j (lanes 0..15 load K pages,
  // lanes 16..31 the same pages for V).  -1 when the lane has nothing to load.
  auto stage_page = [&](int j) -> int32_t {
    if (j >= g.n_stages) return -1;
    const StageGeom s = stage_geom(g, j, ps);
    const int t = lane & 15;
    if (t >= s.npages) return -1;
    return __ldg(p.indices + g.slot_base + s.slot + t);
  };
  auto issue = [&](int j, int slot, int32_t page) {
    const StageGeom s = stage_geom(g, j, ps);
    uint64_t* bar = &mybar[slot];
    T* kdst = mystages + (size_t)slot * 2 * SIDE;
    if (lane == 0) mbar_arrive_expect_tx(bar, 2u * s.npages * box_rows * D * sizeof(T));
    __syncwarp();
    const int t = lane & 15;
    if (t < s.npages) {
      // an out-of-range page id is recorded and redirected past the pool's end,
      // where TMA zero-fills the box instead of reading
      int row = (int)(p.num_pages * ps);
      if ((int64_t)page >= p.num_pages || page < 0) report(p.status, PA_DEVICE_BAD_PAGE);
      else row = page * ps + s.row0;
      T* dst = kdst + (lane < 16 ? 0 : SIDE) + t * box_rows * D;
      tma_load_3d(dst, lane < 16 ? &tm_k : &tm_v, bar, 0, kvh, row, policy);
    }
  };

  // ---- prologue: fill the ring ----
#pragma unroll
  for (int s = 0; s < NSW; ++s) {
    const int j = warp + s * kWarps;
    if (j < g.n_stages) issue(j, s, stage_page(j));
  }
  int32_t next_page = stage_page(warp + NSW * kWarps);

  // ---- queries of the group, pre-scaled into base 2 ----
  float qf[HP][VEC];
#pragma unroll
  for (int h = 0; h < HP; ++h) {
    if (h < nheads) {
      const float* qp = p.q + q_row(p, r, h_first + h) * D + dl * VEC;
#pragma unroll
      for (int e = 0; e < VEC; e += 4) {
        float4 v = *reinterpret_cast<const float4*>(qp + e);
        qf[h][e] = v.x * p.scale_log2;
        qf[h][e + 1] = v.y * p.scale_log2;
        qf[h][e + 2] = v.z * p.scale_log2;
        qf[h][e + 3] = v.w * p.scale_log2;
      }
    } else {
#pragma unroll
      for (int e = 0; e < VEC; ++e) qf[h][e] = 0.f;
    }
  }


  float acc[HP][VEC];
#pragma unroll
  for (int h = 0; h < HP; ++h)
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[h][e] = 0.f;
  float m_run = -INFINITY;  // running max (base 2) of head hs
  float l_run = 0.f;        // running denominator of head hs over this lane's rows
  bool failed = false;

  int i = 0;
  for (;; ++i) {
    const int j = warp + i * kWarps;
    if (j >= g.n_stages) break;
    const int slot = i % NSW;
    if (!mbar_wait_bounded(&mybar[slot], (i / NSW) & 1, kWaitLimitCycles)) {
      failed = true;
      break;
    }
    const StageGeom sg = stage_geom(g, j, ps);
    const T* kb = mystages + (size_t)slot * 2 * SIDE;
    const T* vb = kb + SIDE;

    if (sg.hi > sg.lo) {
      // scores of this lane's head for rows st*TPW + tl
      float s[NSTEP];
#pragma unroll
      for (int st = 0; st < NSTEP; ++st) {
        const int row = st * TPW + tl;
        s[st] = -INFINITY;
        if (st * TPW < sg.hi && st * TPW + TPW > sg.lo) {  // warp-uniform
          float kf[VEC];
          KV<T>::load(kb + row * D + dl * VEC, kf);
          float part[HP];
#pragma unroll
          for (int h = 0; h < HP; ++h) {
            float a = 0.f;
#pragma unroll
            for (int e = 0; e < VEC; ++e) a = fmaf(qf[h][e], kf[e], a);
            part[h] = a;
          }
          const float sc = reduce_scatter<HP, LPT>(part, dl);
          if (row >= sg.lo && row < sg.hi) s[st] = sc;
        }
      }
      // stage max of head hs across the rows of the warp step
      float mt = s[0];
#pragma unroll
      for (int st = 1; st < NSTEP; ++st) mt = fmaxf(mt, s[st]);
#pragma unroll
      for (int o = LPT; o < 32; o <<= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
      const float m_new = fmaxf(m_run, mt);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = fast_exp2(m_run - m_use);
      m_run = m_new;
      float lsum = 0.f;
#pragma unroll
      for (int st = 0; st < NSTEP; ++st) {
        s[st] = fast_exp2(s[st] - m_use);  // becomes p; masked rows give 0
        lsum += s[st];
      }
      l_run = l_run * alpha + lsum;
#pragma unroll
      for (int h = 0; h < HP; ++h) {
        const float a = __shfl_sync(0xffffffffu, alpha, h * LPH);
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[h][e] *= a;
      }
      // P @ V
#pragma unroll
      for (int st = 0; st < NSTEP; ++st) {
        const int row = st * TPW + tl;
        if (st * TPW < sg.hi && st * TPW + TPW > sg.lo) {  // warp-uniform
          float vf[VEC];
          KV<T>::load(vb + row * D + dl * VEC, vf);
          if (!(st * TPW >= sg.lo && st * TPW + TPW <= sg.hi)) {  // partially valid step
            const bool ok = row >= sg.lo && row < sg.hi;
#pragma unroll
            for (int e = 0; e < VEC; ++e) vf[e] = ok ? vf[e] : 0.f;
          }
#pragma unroll
          for (int h = 0; h < HP; ++h) {
            const float ph = __shfl_sync(0xffffffffu, s[st], tl * LPT + h * LPH);
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[h][e] = fmaf(ph, vf[e], acc[h][e]);
          }
        }
      }
    }

    // refill this slot with the warp's stage NSW rounds ahead
    __syncwarp();
    const int jn = warp + (i + NSW) * kWarps;
    if (jn < g.n_stages) {
      fence_proxy_async_smem();
      issue(jn, slot, next_page);
      next_page = stage_page(jn + kWarps);
    }
  }

  if (failed) {
    if (lane == 0) report(p.status, PA_DEVICE_WAIT_TIMEOUT);
    // drain this warp's copies still in flight before the CTA's shared memory is reused
    for (int k = i + 1; k < i + NSW; ++k) {
      if (warp + k * kWarps >= g.n_stages) break;
      mbar_wait_bounded(&mybar[k % NSW], (k / NSW) & 1, kWaitLimitCycles);
    }
  }

  // ---- combine the rows of the warp step, then the warps ----
#pragma unroll
  for (int o = LPT; o < 32; o <<= 1) {
    l_run += __shfl_xor_sync(0xffffffffu, l_run, o);
#pragma unroll
    for (int h = 0; h < HP; ++h)
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], o);
  }
  __syncthreads();  // every warp is done with its stages: reuse them for the states
  if (tl == 0) {
#pragma unroll
    for (int h = 0; h < HP; ++h)
#pragma unroll
      for (int e = 0; e < VEC; ++e) accs[(warp * HP + h) * D + dl * VEC + e] = acc[h][e];
    if (dl % LPH == 0) {
      ms[warp * HP + hs] = m_run;
      ls[warp * HP + hs] = l_run;
    }
  }
  __syncthreads();
  finish_chunk<HP, D, kWarps>(p, g, ms, ls, accs, accs, c, r, h_first, nheads);
}

// ---- host side --------------------------------------------------------------

using SimtKernel = void (*)(const CUtensorMap, const CUtensorMap, const PartialParams);

template <typename T, int D>
constexpr int simt_ring_depth() {
  return (sizeof(T) * 2 * kStageRows * D) <= 8192 ? 3 : 2;
}

template <typename T, int D, int HP>
size_t simt_smem_bytes() {
  constexpr int NSW = simt_ring_depth<T, D>();
  size_t stage = sizeof(T) * kWarps * NSW * 2 * kStageRows * D;
  size_t states = sizeof(float) * kWarps * HP * D;
  size_t body = stage > states ? stage : states;
  return body + sizeof(uint64_t) * kWarps * NSW + 2 * sizeof(float) * kWarps * HP;
}

struct SimtInstance {
  SimtKernel fn;
  size_t smem;
};

template <typename T, int D, int HP>
SimtInstance simt_make() {
  return {pa_v2_partial_simt_kernel<T, D, HP, simt_ring_depth<T, D>()>, simt_smem_bytes<T, D, HP>()};
}

template <typename T, int D>
bool simt_pick_hp(int hp, SimtInstance* out) {
  switch (hp) {
    case 1: *out = simt_make<T, D, 1>(); return true;
    case 2: *out = simt_make<T, D, 2>(); return true;
    case 4: *out = simt_make<T, D, 4>(); return true;
    case 8: *out = simt_make<T, D, 8>(); return true;
    default: return false;
  }
}

bool simt_pick(int dtype, int D, int hpc, SimtInstance* out) {
  int hp = 1;
  while (hp < hpc) hp <<= 1;
  if (D == 64) {
    if (dtype == PA_F32) return simt_pick_hp<float, 64>(hp, out);
    if (dtype == PA_F16) return simt_pick_hp<__half, 64>(hp, out);
    if (dtype == PA_BF16) return simt_pick_hp<__nv_bfloat16, 64>(hp, out);
  } else if (D == 128) {
    if (dtype == PA_F32) return simt_pick_hp<float, 128>(hp, out);
    if (dtype == PA_F16) return simt_pick_hp<__half, 128>(hp, out);
    if (dtype == PA_BF16) return simt_pick_hp<__nv_bfloat16, 128>(hp, out);
  }
  return false;
}

}  // namespace

int launch_partial_simt(const LaunchArgs& a) {
  SimtInstance inst;
  if (!simt_pick(a.kv_dtype, a.head_dim, a.p.hpc, &inst)) return PA_EUNSUPPORTED;
  if (!prepare_kernel(reinterpret_cast<const void*>(inst.fn), inst.smem)) return PA_ECUDA;
  dim3 grid(a.num_chunks, a.p.num_kv_heads * a.p.q_groups);
  const cudaError_t rc = launch_dependent(inst.fn, grid, dim3(kWarps * 32), inst.smem, a.stream, *a.tm_k, *a.tm_v, a.p);
  return rc == cudaSuccess && cudaGetLastError() == cudaSuccess ? PA_OK : PA_ECUDA;
}

int occupancy_partial_simt(int kv_dtype, int head_dim, int hpc, int* blocks_per_sm) {
  SimtInstance inst;
  if (!simt_pick(kv_dtype, head_dim, hpc, &inst)) return PA_EUNSUPPORTED;
  if (!prepare_kernel(reinterpret_cast<const void*>(inst.fn), inst.smem)) return PA_ECUDA;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, inst.fn, kWarps * 32, inst.smem) ==
                 cudaSuccess
             ? PA_OK
             : PA_ECUDA;
}

}  // namespace pa
