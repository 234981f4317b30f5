// pa_partial_tc.cu -- tensor-core variant of the split-KV partial kernel (f16 / bf16 pools).
//
// Same contract as the CUDA-core variant (issue #898 "Fused paged-attention
// decode v2: CSR page table, cross-CTA split-KV, and variable-length merge
// kernels", design pieces 1-2; PR #984 "fused paged-attention decode v2 with
// CSR page table and cross-CTA split-KV", What changed 2): one CTA per (chunk,
// kv head, q-head group), each K/V element read once for the whole group, an
// online softmax in base 2, a normalized partial and its log2-LSE per chunk.
//
// Why tensor cores here.  Decode attention is HBM-bound, but with a GQA group
// of 4-16 heads a CUDA-core mapping spends ~1.5k warp instructions per 16
// tokens on FMAs, conversions and shuffle reductions, which keeps the SM
// issue-bound below the HBM roofline.  Per 16-token stage this kernel instead
// issues two m16n8k16 MMAs per 16 head-dims for Q.K and two per 16 head-dims
// for P.V (warp-level mma.sync), each fed by one ldmatrix:
//
//   S^T [16 tokens x 8 heads] = K [16 x D] . Q^T [D x 8]          (tokens are M)
//   O^T [D x 8 heads]        += V^T [D x 16] . P^T [16 x 8]
//
// The K/V stage is 16 rows of one KV head stored as 128-byte half rows with
// the 16-byte chunk index XOR-ed by (row mod 8) -- the layout TMA's 128-byte
// swizzle writes -- so every ldmatrix phase touches 8 distinct bank groups.
// Q and P enter the MMA as hi + lo pairs of the pool's 16-bit type (x = hi +
// lo with hi = round(x), lo = round(x - hi)): products of the exact 16-bit K/V
// values with both halves accumulate in f32, which keeps the scores and the
// output at f32-level accuracy instead of the 2^-9 (bf16) rounding of a single
// 16-bit operand.
//
// Staging: TMA (cp.async.bulk.tensor with SWIZZLE_128B, completion on an
// mbarrier) when pages start on 8-row boundaries of a stage (page_size 8, 16
// or a multiple of 16); otherwise cp.async 16-byte copies that apply the same
// swizzle in the destination address, with the row -> (page, entry) split done
// by a fast division by page_size.
#include "pa_partial_tc_body.cuh"

namespace pa {
namespace {

template <typename T, int D, int NT, int NSW, int NW, bool USE_TMA>
__global__ void __launch_bounds__(NW * 32)
    pa_v2_partial_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                            const PartialParams p) {
  partial_tc_body<T, D, NT, NSW, NW, USE_TMA>(tm_k, tm_v, p, blockIdx.x, blockIdx.y, -1, -1);
}

// ---- host side --------------------------------------------------------------

using TcKernel = void (*)(const CUtensorMap, const CUtensorMap, const PartialParams);

struct TcInstance {
  TcKernel fn;
  size_t smem;
};

template <typename T, int D, int NT, bool TMA>
TcInstance tc_make() {
  return {pa_v2_partial_tc_kernel<T, D, NT, kTcRing, kTcWarps, TMA>,
          (size_t)TcLayout<D, NT, kTcRing, kTcWarps>::ALLOC};
}

template <typename T, int D, bool TMA>
bool tc_pick_nt(int hpc, TcInstance* out) {
  if (hpc <= 8) { *out = tc_make<T, D, 1, TMA>(); return true; }
  if (hpc <= 16) { *out = tc_make<T, D, 2, TMA>(); return true; }
  return false;
}

template <typename T, int D>
bool tc_pick_stage(int hpc, bool tma, TcInstance* out) {
  return tma ? tc_pick_nt<T, D, true>(hpc, out) : tc_pick_nt<T, D, false>(hpc, out);
}

bool tc_pick(int dtype, int D, int hpc, bool tma, TcInstance* out) {
  if (dtype == PA_F16) {
    if (D == 64) return tc_pick_stage<__half, 64>(hpc, tma, out);
    if (D == 128) return tc_pick_stage<__half, 128>(hpc, tma, out);
  } else if (dtype == PA_BF16) {
    if (D == 64) return tc_pick_stage<__nv_bfloat16, 64>(hpc, tma, out);
    if (D == 128) return tc_pick_stage<__nv_bfloat16, 128>(hpc, tma, out);
  }
  return false;
}

}  // namespace

int launch_partial_tc(const LaunchArgs& a, bool use_tma) {
  TcInstance inst;
  if (!tc_pick(a.kv_dtype, a.head_dim, a.p.hpc, use_tma, &inst)) return PA_EUNSUPPORTED;
  if (!prepare_kernel(reinterpret_cast<const void*>(inst.fn), inst.smem)) return PA_ECUDA;
  dim3 grid(a.num_chunks, a.p.num_kv_heads * a.p.q_groups);
  const cudaError_t rc = launch_dependent(inst.fn, grid, dim3(kTcWarps * 32), inst.smem, a.stream, *a.tm_k, *a.tm_v, a.p);
  return rc == cudaSuccess && cudaGetLastError() == cudaSuccess ? PA_OK : PA_ECUDA;
}

int occupancy_partial_tc(int kv_dtype, int head_dim, int hpc, bool use_tma, int* blocks_per_sm) {
  TcInstance inst;
  if (!tc_pick(kv_dtype, head_dim, hpc, use_tma, &inst)) return PA_EUNSUPPORTED;
  if (!prepare_kernel(reinterpret_cast<const void*>(inst.fn), inst.smem)) return PA_ECUDA;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, inst.fn, kTcWarps * 32, inst.smem) ==
                 cudaSuccess
             ? PA_OK
             : PA_ECUDA;
}

}  // namespace pa
