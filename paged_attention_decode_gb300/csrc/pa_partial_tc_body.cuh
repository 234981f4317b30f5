// pa_partial_tc_body.cuh -- the body of the tensor-core split-KV partial kernel
// (f16 / bf16 pools), shared by the one-plan kernel (pa_partial_tc.cu) and the
// kernel that runs the two cascade levels in one launch
// (pa_partial_tc_cascade.cu).  The design notes are at the top of
// pa_partial_tc.cu.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "pa_internal.cuh"
#include "pa_mma.cuh"

namespace pa {

constexpr int kTcRing = 3;   // stages in flight per warp
constexpr int kTcWarps = 8;  // one CTA of 8 warps per SM: 8 x 3 x 8 KB of stages

// ---- the kernel -------------------------------------------------------------

template <int D, int NT, int NSW, int NW>
struct TcLayout {
  static constexpr int HP = 8 * NT;                 // query heads per CTA (padded)
  static constexpr int TILE = (D / 64) * 2048;       // bytes of one side of a stage
  static constexpr int STAGE = 2 * TILE;
  static constexpr int STAGES_BYTES = NW * NSW * STAGE;
  static constexpr int PT_BYTES = NW * 2 * HP * 32;   // P^T hi/lo per warp: [HP][16] 16-bit
  static constexpr int DP = D + 4;                   // state row stride: 4 floats of padding per row
  static constexpr int STATE_BYTES = NW * HP * DP * 4;
  static constexpr int BODY = STAGES_BYTES > STATE_BYTES ? STAGES_BYTES : STATE_BYTES;
  static constexpr int BARS = BODY + PT_BYTES;
  static constexpr int MS = BARS + NW * NSW * 8;
  static constexpr int TOTAL = MS + 2 * NW * HP * 4;
  static constexpr int ALLOC = TOTAL + 1024;         // room to align the base to 1 KB
};

// T: __half or __nv_bfloat16.  D: 64 or 128.  NT: 8-head n-tiles per CTA (1 or
// 2).  NSW: stage ring depth per warp.  NW: warps per CTA.  USE_TMA: staging
// mechanism.
//
// The body runs chunk c of plan p as CTA row y of ny (the CTAs of one chunk: KV heads x q-groups) in a
// launch whose plan has num_chunks chunks (-1 for y, num_chunks, ny: this grid's own).
template <typename T, int D, int NT, int NSW, int NW, bool USE_TMA, bool MAPPED = false>
__device__ __forceinline__ void partial_tc_body(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                                const PartialParams& p, const int c, const int y,
                                                const int num_chunks, const int ny) {
  using L = TcLayout<D, NT, NSW, NW>;
  constexpr int HP = L::HP;
  // EARLY: copy a stage's K and V fragments to registers and release its slot
  // before the math.  Measured slower on GB300 (26.9 vs 26.1 us on the 32K
  // decode, same GPU), so the slot is released after the math.
  constexpr bool EARLY = false;
  constexpr int KSTEPS = D / 16;
  constexpr int CPR = D / 8;  // 16-byte chunks per K/V row

  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BARS);
  float* ms = reinterpret_cast<float*>(smem + L::MS);
  float* ls = ms + NW * HP;
  float* accs = reinterpret_cast<float*>(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;  // MMA group row
  const int t = lane & 3;   // MMA thread-in-group
  const int kvh = y / p.q_groups;
  const int qg = y % p.q_groups;
  const int h_first = kvh * p.group + qg * p.hpc;
  const int nheads = min(p.hpc, p.group - qg * p.hpc);
  const int ps = p.page_size;

  // the kernel that follows (the merge, or the next step) may be scheduled now;
  // it waits for this grid to finish
  pdl_launch_dependents();

  // the warp's stage barriers: shared memory only, so set up while the kernel
  // before this one may still be running
  uint64_t* mybar = bars + warp * NSW;
  if (USE_TMA) {
    if (lane == 0) {
#pragma unroll
      for (int s = 0; s < NSW; ++s) mbar_init(&mybar[s], 1);
      fence_barrier_init();
    }
    __syncwarp();
  }

  // Before the wait, while the kernel before this one may still be running
  // (its last CTAs, or the merge of the step before): warm L2 with this warp's
  // first stage, from a speculative read of the chunk geometry and of the
  // stage's page ids.  Nothing read here reaches the result -- values are
  // bounds-checked and only choose prefetch addresses -- and all of it is read
  // again after the wait; the stage's loads then find their rows in L2 instead
  // of waiting out a DRAM round trip behind the page-id load.  Lines are
  // prefetched from the load/store path, leaving the TMA unit to the stages'
  // loads.  One stage, not the ring's NSW: when nothing runs before this
  // kernel the prefetches are still in flight as the stages' own loads go out,
  // and prefetching NSW stages cost such a launch 2-4 us on GB300.  The host
  // sets warm_l2 where the chain ahead of the prefetches is short (see
  // prepare_decode).
  if (p.warm_l2) {
    int rs;
    const ChunkGeom sg = chunk_geom<true>(p, c, &rs);
    if (warp < sg.n_stages) {  // warp-uniform
      const StageGeom st = stage_geom(sg, warp, ps);
      const int tp = lane & 15;  // row (tp) of the stage; K for lanes 0-15, V for 16-31
      const int32_t pg = tp < st.npages ? __ldcg(p.indices + sg.slot_base + st.slot + tp) : -1;
      const int sl = (int)fast_div((uint32_t)tp, p.ps_magic, p.ps_shift);  // page of row tp within the stage
      const int32_t page = __shfl_sync(0xffffffffu, pg, sl & 15);
      const int rows = ps <= kStageRows ? st.npages * ps : kStageRows;
      if (tp < rows && page >= 0 && (int64_t)page < p.num_pages) {
        constexpr int ROW_BYTES = D * (int)sizeof(T);
        const unsigned char* pool = static_cast<const unsigned char*>(lane >= 16 ? p.v_pool : p.k_pool);
        const unsigned char* a =
            pool + (((size_t)page * ps + st.row0 + (tp - sl * ps)) * p.num_kv_heads + kvh) * ROW_BYTES;
#pragma unroll
        for (int b = 0; b < ROW_BYTES; b += 128) prefetch_l2(a + b);
      }
    }
  }

  // launched as a programmatic dependent: the kernel before this one in the
  // stream has completed, and its writes are visible, once this returns
  pdl_wait_prerequisites();

  int r;
  const ChunkGeom gm = chunk_geom(p, c, &r);

  unsigned char* mst = smem + warp * NSW * L::STAGE;
  unsigned short* pt_hi = reinterpret_cast<unsigned short*>(smem + L::BODY + warp * 2 * HP * 32);
  unsigned short* pt_lo = pt_hi + HP * 16;
  const uint64_t policy = policy_evict_first();
  const int box_rows = ps <= kStageRows ? ps : kStageRows;

  // ---- staging ----
  // Lane (lane & 15) holds the page id of page (lane & 15) of stage j, or -1.
  auto stage_page = [&](int j) -> int32_t {
    if (j >= gm.n_stages) return -1;
    const StageGeom s = stage_geom(gm, j, ps);
    const int tp = lane & 15;
    if (tp >= s.npages) return -1;
    return __ldg(p.indices + gm.slot_base + s.slot + tp);
  };
  auto page_ok = [&](int32_t page) { return page >= 0 && (int64_t)page < p.num_pages; };

  auto issue_tma = [&](int j, int slot, int32_t my_page) {
    const StageGeom s = stage_geom(gm, j, ps);
    constexpr int HALVES = D / 64;
    const int nops = s.npages * HALVES * 2;
    const int tp = lane / (2 * HALVES);
    const int32_t page = __shfl_sync(0xffffffffu, my_page, tp & 15);
    uint64_t* bar = &mybar[slot];
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(nops * box_rows * 128));
    __syncwarp();
    if (lane < nops) {
      const int side = (lane / HALVES) & 1;
      const int half = lane % HALVES;
      int row = (int)(p.num_pages * ps);  // past the pool's end: TMA zero-fills
      if (page_ok(page)) row = page * ps + s.row0;
      else report(p.status, PA_DEVICE_BAD_PAGE);
      unsigned char* dst = mst + slot * L::STAGE + side * L::TILE + half * 2048 + tp * box_rows * 128;
      tma_load_3d(dst, side ? &tm_v : &tm_k, bar, half * 64, kvh, row, policy);
    }
  };

  auto issue_cpasync = [&](int j, int slot, int32_t my_page) {
    const StageGeom s = stage_geom(gm, j, ps);
    const int nrows = s.npages * ps;
    constexpr int RSTEP = 32 / CPR;
    const int ch = lane % CPR;
    const int r0 = lane / CPR;
    const uint32_t kdst = smem_addr(mst + slot * L::STAGE);
    const uint32_t vdst = kdst + L::TILE;
    const T* kp = static_cast<const T*>(p.k_pool);
    const T* vp = static_cast<const T*>(p.v_pool);
#pragma unroll
    for (int i = 0; i < kStageRows / RSTEP; ++i) {
      const int row = r0 + i * RSTEP;
      const int sl = (int)fast_div((uint32_t)row, p.ps_magic, p.ps_shift);  // row / page_size
      const int e = row - sl * ps;
      const int32_t page = __shfl_sync(0xffffffffu, my_page, sl & 15);
      if (row < nrows) {
        if (page_ok(page)) {
          const size_t elem = (((size_t)page * ps + e) * p.num_kv_heads + kvh) * D + ch * 8;
          const uint32_t off = swz(row, ch);
          cp_async_16(kdst + off, kp + elem, policy);
          cp_async_16(vdst + off, vp + elem, policy);
        } else {
          report(p.status, PA_DEVICE_BAD_PAGE);
        }
      }
    }
  };

  auto issue = [&](int j, int slot, int32_t my_page) {
    if (USE_TMA) issue_tma(j, slot, my_page);
    else issue_cpasync(j, slot, my_page);
  };

#pragma unroll
  for (int s = 0; s < NSW; ++s) {
    const int j = warp + s * NW;
    if (j < gm.n_stages) issue(j, s, stage_page(j));
    if (!USE_TMA) cp_async_commit();
  }
  int32_t next_page = stage_page(warp + NSW * NW);

  // ---- Q fragments (loaded while the first stages stream in): B operand of
  // S^T = K Q^T, base-2 scaled, split hi + lo ----
  uint32_t qh[KSTEPS][NT][2], ql[KSTEPS][NT][2];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int head = 8 * j + g;
    const bool ok = head < nheads;
    const float* qp = p.q + q_row(p, r, h_first + (ok ? head : 0)) * D + 2 * t;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      float x[4];
      x[0] = ok ? qp[16 * kk] * p.scale_log2 : 0.f;
      x[1] = ok ? qp[16 * kk + 1] * p.scale_log2 : 0.f;
      x[2] = ok ? qp[16 * kk + 8] * p.scale_log2 : 0.f;
      x[3] = ok ? qp[16 * kk + 9] * p.scale_log2 : 0.f;
      float h[4], l[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        h[e] = TC<T>::round(x[e]);
        l[e] = x[e] - h[e];
      }
      qh[kk][j][0] = TC<T>::pack(h[0], h[1]);
      qh[kk][j][1] = TC<T>::pack(h[2], h[3]);
      ql[kk][j][0] = TC<T>::pack(l[0], l[1]);
      ql[kk][j][1] = TC<T>::pack(l[2], l[3]);
    }
  }


  float o[KSTEPS][NT][4];
#pragma unroll
  for (int mt = 0; mt < KSTEPS; ++mt)
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mt][j][e] = 0.f;
  float m_run[NT][2], l_run[NT][2];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    m_run[j][0] = m_run[j][1] = -INFINITY;
    l_run[j][0] = l_run[j][1] = 0.f;
  }
  bool failed = false;

  int i = 0;
  for (;; ++i) {
    const int j = warp + i * NW;
    if (j >= gm.n_stages) break;
    const int slot = i % NSW;
    if (USE_TMA) {
      if (!mbar_wait_bounded(&mybar[slot], (i / NSW) & 1, kWaitLimitCycles)) {
        failed = true;
        break;
      }
    } else {
      cp_async_wait<NSW - 1>();
      __syncwarp();
    }
    const StageGeom sg = stage_geom(gm, j, ps);
    unsigned char* kt = mst + slot * L::STAGE;
    unsigned char* vt = kt + L::TILE;
    const uint32_t kbase = smem_addr(kt);
    const uint32_t vbase = smem_addr(vt);
    const int krow = ((lane >> 3) & 1) * 8 + (lane & 7);  // K fragment row this lane addresses
    const int vtok = (lane >> 4) * 8 + (lane & 7);        // V^T fragment token this lane addresses

    // rows of the V tile outside [lo, hi) may hold stale or non-finite data: zero them
    if (sg.lo > 0 || sg.hi < kStageRows) {
      for (int idx = lane; idx < kStageRows * CPR; idx += 32) {
        const int row = idx / CPR;
        if (row < sg.lo || row >= sg.hi)
          *reinterpret_cast<uint4*>(vt + (idx % CPR >> 3) * 2048 + row * 128 + (idx % 8) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
    }

    // Refill this slot with the warp's stage NSW rounds ahead (after the math,
    // or, with EARLY, once the stage's fragments are in registers).
    auto refill = [&]() {
      const int jn = warp + (i + NSW) * NW;
      if (jn < gm.n_stages) {
        if (USE_TMA) fence_proxy_async_smem();
        issue(jn, slot, next_page);
        next_page = stage_page(jn + NW);
      }
      if (!USE_TMA) cp_async_commit();
    };
    uint32_t kf[EARLY ? KSTEPS : 1][4], vf[EARLY ? KSTEPS : 1][4];
    if (EARLY) {
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) ldsm_x4(kf[kk], kbase + swz(krow, kk * 2 + (lane >> 4)));
#pragma unroll
      for (int mt = 0; mt < KSTEPS; ++mt) ldsm_x4_trans(vf[mt], vbase + swz(vtok, mt * 2 + ((lane >> 3) & 1)));
      __syncwarp();  // every lane's shared-memory reads of the slot are done
      refill();
    }

    // ---- S^T = K . Q^T: hi and lo halves, even and odd k-steps in separate accumulators ----
    float sacc[4][NT][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int jj = 0; jj < NT; ++jj)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[a][jj][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      uint32_t a[4];
      if (EARLY) {
#pragma unroll
        for (int e = 0; e < 4; ++e) a[e] = kf[kk][e];
      } else {
        ldsm_x4(a, kbase + swz(krow, kk * 2 + (lane >> 4)));
      }
#pragma unroll
      for (int jj = 0; jj < NT; ++jj) {
        TC<T>::mma(sacc[kk & 1][jj], a, qh[kk][jj][0], qh[kk][jj][1]);
        TC<T>::mma(sacc[2 + (kk & 1)][jj], a, ql[kk][jj][0], ql[kk][jj][1]);
      }
    }

    // ---- online softmax over the stage (tokens g and g + 8, heads 2t, 2t + 1) ----
    const bool v0 = g >= sg.lo && g < sg.hi;
    const bool v1 = g + 8 >= sg.lo && g + 8 < sg.hi;
    float pr[NT][4];
#pragma unroll
    for (int jj = 0; jj < NT; ++jj) {
      float sv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) sv[e] = (sacc[0][jj][e] + sacc[1][jj][e]) + (sacc[2][jj][e] + sacc[3][jj][e]);
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
      const float mn0 = fmaxf(m_run[jj][0], mx0), mn1 = fmaxf(m_run[jj][1], mx1);
      const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
      const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
      const float a0 = fast_exp2(m_run[jj][0] - mu0), a1 = fast_exp2(m_run[jj][1] - mu1);
      m_run[jj][0] = mn0;
      m_run[jj][1] = mn1;
      pr[jj][0] = fast_exp2(s0 - mu0);
      pr[jj][1] = fast_exp2(s1 - mu1);
      pr[jj][2] = fast_exp2(s2 - mu0);
      pr[jj][3] = fast_exp2(s3 - mu1);
      l_run[jj][0] = l_run[jj][0] * a0 + pr[jj][0] + pr[jj][2];
      l_run[jj][1] = l_run[jj][1] * a1 + pr[jj][1] + pr[jj][3];
#pragma unroll
      for (int mt = 0; mt < KSTEPS; ++mt) {
        o[mt][jj][0] *= a0;
        o[mt][jj][1] *= a1;
        o[mt][jj][2] *= a0;
        o[mt][jj][3] *= a1;
      }
      // P^T [head][token] for the B operand, hi and lo
      const int h0 = 8 * jj + 2 * t;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int hh = h0 + (e & 1);
        const int tok = g + (e >> 1) * 8;
        const float hi = TC<T>::round(pr[jj][e]);
        pt_hi[hh * 16 + tok] = TC<T>::bits(hi);
        pt_lo[hh * 16 + tok] = TC<T>::bits(pr[jj][e] - hi);
      }
    }
    __syncwarp();

    // ---- O^T += V^T . P^T ----
    uint32_t bph[NT][2], bpl[NT][2];
#pragma unroll
    for (int jj = 0; jj < NT; ++jj) {
      const unsigned short* src = (lane >> 4) ? pt_lo : pt_hi;
      const int head = 8 * jj + (lane & 7);
      const int tokoff = ((lane >> 3) & 1) * 8;
      uint32_t b[4];
      ldsm_x4(b, smem_addr(src + head * 16 + tokoff));
      bph[jj][0] = b[0];
      bph[jj][1] = b[1];
      bpl[jj][0] = b[2];
      bpl[jj][1] = b[3];
    }
#pragma unroll
    for (int mt = 0; mt < KSTEPS; ++mt) {
      uint32_t a[4];
      if (EARLY) {
#pragma unroll
        for (int e = 0; e < 4; ++e) a[e] = vf[mt][e];
      } else {
        ldsm_x4_trans(a, vbase + swz(vtok, mt * 2 + ((lane >> 3) & 1)));
      }
#pragma unroll
      for (int jj = 0; jj < NT; ++jj) {
        TC<T>::mma(o[mt][jj], a, bph[jj][0], bph[jj][1]);
        TC<T>::mma(o[mt][jj], a, bpl[jj][0], bpl[jj][1]);
      }
    }
    __syncwarp();  // the P^T buffer is rewritten by the next stage
    if (!EARLY) refill();
  }

  if (USE_TMA) {
    if (failed) {
      if (lane == 0) report(p.status, PA_DEVICE_WAIT_TIMEOUT);
      for (int k = i + 1; k < i + NSW; ++k) {
        if (warp + k * NW >= gm.n_stages) break;
        mbar_wait_bounded(&mybar[k % NSW], (k / NSW) & 1, kWaitLimitCycles);
      }
    }
  } else {
    cp_async_wait<0>();
  }

  // ---- per-warp state -> shared memory, then merge the warps ----
#pragma unroll
  for (int jj = 0; jj < NT; ++jj)
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) l_run[jj][e] += __shfl_xor_sync(0xffffffffu, l_run[jj][e], off);
  __syncthreads();  // all warps are done with their stages: reuse them for the states
#pragma unroll
  for (int mt = 0; mt < KSTEPS; ++mt)
#pragma unroll
    for (int jj = 0; jj < NT; ++jj) {
      const int h0 = 8 * jj + 2 * t;
      // rows DP = D + 4 floats apart: the four t-lanes writing rows h0 = 2t land in distinct banks
      float* a0 = accs + (warp * HP + h0) * L::DP + 16 * mt + g;
      float* a1 = a0 + L::DP;
      a0[0] = o[mt][jj][0];
      a1[0] = o[mt][jj][1];
      a0[8] = o[mt][jj][2];
      a1[8] = o[mt][jj][3];
    }
  if (g == 0) {
#pragma unroll
    for (int jj = 0; jj < NT; ++jj) {
      const int h0 = 8 * jj + 2 * t;
      ms[warp * HP + h0] = m_run[jj][0];
      ms[warp * HP + h0 + 1] = m_run[jj][1];
      ls[warp * HP + h0] = l_run[jj][0];
      ls[warp * HP + h0 + 1] = l_run[jj][1];
    }
  }
  __syncthreads();
  finish_chunk<HP, D, NW, MAPPED, L::DP>(p, gm, ms, ls, accs, accs, c, r, h_first, nheads, num_chunks, y, ny);
}

}  // namespace pa
