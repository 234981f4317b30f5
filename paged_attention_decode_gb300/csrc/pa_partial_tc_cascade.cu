// pa_partial_tc_cascade.cu -- the two cascade levels in one launch of the
// tensor-core partial kernel (cascade-attention.md, issue #903, composition and
// head-stacking paragraphs): CTA columns [0, split) run level 0's chunks (the
// members' heads stacked over the shared pages), the rest level 1's.  Kept in
// its own translation unit so that the one-plan kernel's module is unchanged.
#include "pa_partial_tc_body.cuh"

namespace pa {
namespace {

// Two plans over the same pools in one launch (the two cascade levels, cascade-attention.md): CTA columns
// [0, split) run plan p0's chunks, the rest plan p1's (n1 chunks); a CTA whose row is past its plan's CTAs
// per chunk leaves before touching memory.  Each plan writes its partials (and merges, when fused) as its own
// launch would, with its own n-tile count: level 0's CTAs carry the members' stacked heads (NT0 8-head
// tiles), level 1's only a request's (NT1), so a level-1 CTA does not pay for level 0's empty columns.
template <typename T, int D, int NT0, int NT1, int NSW, int NW, bool USE_TMA>
__global__ void __launch_bounds__(NW * 32)
    pa_v2_partial_tc_two_plan_kernel(const __grid_constant__ CUtensorMap tm_k,
                                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ PartialParams p0,
                                     const __grid_constant__ PartialParams p1, const int split, const int n1) {
  if ((int)blockIdx.x < split) {
    const int ny = p0.num_kv_heads * p0.q_groups;
    if ((int)blockIdx.y < ny)
      partial_tc_body<T, D, NT0, NSW, NW, USE_TMA, true>(tm_k, tm_v, p0, blockIdx.x, blockIdx.y, split, ny);
  } else {
    const int ny = p1.num_kv_heads * p1.q_groups;
    if ((int)blockIdx.y < ny)
      partial_tc_body<T, D, NT1, NSW, NW, USE_TMA, true>(tm_k, tm_v, p1, blockIdx.x - split, blockIdx.y, n1, ny);
  }
}

using TcKernel2 = void (*)(const CUtensorMap, const CUtensorMap, const PartialParams, const PartialParams, const int,
                           const int);

struct Tc2Instance {
  TcKernel2 fn;
  size_t smem;
};

template <typename T, int D, int NT0, int NT1, bool TMA>
Tc2Instance tc2_make() {
  constexpr size_t a0 = TcLayout<D, NT0, kTcRing, kTcWarps>::ALLOC, a1 = TcLayout<D, NT1, kTcRing, kTcWarps>::ALLOC;
  return {pa_v2_partial_tc_two_plan_kernel<T, D, NT0, NT1, kTcRing, kTcWarps, TMA>, a0 > a1 ? a0 : a1};
}

// nt0 >= nt1: level 0 stacks the members' heads over level 1's group
template <typename T, int D, bool TMA>
bool tc2_pick_nt(int nt0, int nt1, Tc2Instance* out) {
  if (nt0 == 1 && nt1 == 1) { *out = tc2_make<T, D, 1, 1, TMA>(); return true; }
  if (nt0 == 2 && nt1 == 1) { *out = tc2_make<T, D, 2, 1, TMA>(); return true; }
  if (nt0 == 2 && nt1 == 2) { *out = tc2_make<T, D, 2, 2, TMA>(); return true; }
  return false;
}

template <typename T, int D>
bool tc2_pick_stage(int nt0, int nt1, bool tma, Tc2Instance* out) {
  return tma ? tc2_pick_nt<T, D, true>(nt0, nt1, out) : tc2_pick_nt<T, D, false>(nt0, nt1, out);
}

// 8-head n-tiles for hpc query heads per CTA (0: more than the kernel serves)
int tc2_tiles(int hpc) { return hpc <= 8 ? 1 : hpc <= 16 ? 2 : 0; }

bool tc2_pick(int dtype, int D, int hpc0, int hpc1, bool tma, Tc2Instance* out) {
  const int nt0 = tc2_tiles(hpc0), nt1 = tc2_tiles(hpc1);
  if (dtype == PA_F16) {
    if (D == 64) return tc2_pick_stage<__half, 64>(nt0, nt1, tma, out);
    if (D == 128) return tc2_pick_stage<__half, 128>(nt0, nt1, tma, out);
  } else if (dtype == PA_BF16) {
    if (D == 64) return tc2_pick_stage<__nv_bfloat16, 64>(nt0, nt1, tma, out);
    if (D == 128) return tc2_pick_stage<__nv_bfloat16, 128>(nt0, nt1, tma, out);
  }
  return false;
}

}  // namespace

int launch_partial_tc_two_plans(const LaunchArgs& a, const PartialParams& p1, int n1, bool use_tma) {
  Tc2Instance inst;
  if (!tc2_pick(a.kv_dtype, a.head_dim, a.p.hpc, p1.hpc, use_tma, &inst)) return PA_EUNSUPPORTED;
  if (!prepare_kernel(reinterpret_cast<const void*>(inst.fn), inst.smem)) return PA_ECUDA;
  const int y0 = a.p.num_kv_heads * a.p.q_groups, y1 = p1.num_kv_heads * p1.q_groups;
  dim3 grid(a.num_chunks + n1, y0 > y1 ? y0 : y1);
  const cudaError_t rc = launch_dependent(inst.fn, grid, dim3(kTcWarps * 32), inst.smem, a.stream, *a.tm_k, *a.tm_v,
                                          a.p, p1, a.num_chunks, n1);
  return rc == cudaSuccess && cudaGetLastError() == cudaSuccess ? PA_OK : PA_ECUDA;
}

}  // namespace pa
