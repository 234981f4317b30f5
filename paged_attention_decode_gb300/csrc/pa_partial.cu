// pa_partial.cu -- C-ABI entry of the split-KV partial kernel: argument checks,
// kernel-variant choice, TMA tensor maps over the pools, launch; the
// q-heads-per-CTA rule; and the occupancy-derived default CTA target of the plan.
//
// Variants (same contract; issue #898 "Fused paged-attention decode v2: CSR
// page table, cross-CTA split-KV, and variable-length merge kernels", design
// piece 2; PR #984 "fused paged-attention decode v2 with CSR page table and
// cross-CTA split-KV", What changed 2):
//  - tensor cores (pa_partial_tc.cu) for f16 / bf16 pools, up to 16 query
//    heads per CTA;
//  - CUDA cores (pa_partial_simt.cu) for f32 pools (or on request through
//    plan.kernel), up to 8 query heads per CTA.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "pa_internal.cuh"
#include "pa_launch.h"

namespace pa {

bool prepare_kernel(const void* fn, size_t smem) {
  constexpr int kMaxDevices = 64;
  constexpr int kMaxKernels = 128;
  static std::mutex mu;
  static const void* done[kMaxDevices][kMaxKernels] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < kMaxKernels; ++i) {
    if (done[dev][i] == fn) return true;
    if (done[dev][i] == nullptr) {
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return false;
      done[dev][i] = fn;
      return true;
    }
  }
  return false;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Tensor map over a pool viewed as [rows = num_pages * page_size, Hkv, D]
// (innermost first: D, Hkv, rows); a box is one KV head x `box_rows` rows x
// `box_d` elements of the head dim.
bool make_pool_map(CUtensorMap* map, const void* base, int dtype, int64_t rows, int hkv, int D, int box_d,
                   int box_rows, CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  const CUtensorMapDataType dt = dtype == PA_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : dtype == PA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int esize = dtype == PA_F32 ? 4 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)hkv, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)D * esize, (cuuint64_t)hkv * D * esize};
  cuuint32_t box[3] = {(cuuint32_t)box_d, 1u, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult rc = fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool use_tensor_cores(int kv_dtype, int kernel) {
  return kernel != 1 && (kv_dtype == PA_F16 || kv_dtype == PA_BF16);
}

}  // namespace
}  // namespace pa

extern "C" int32_t pa_v2_q_heads_per_cta(int32_t group_size, int32_t head_dim, int32_t kv_dtype) {
  if (group_size < 1) return 0;
  if (head_dim == 512)  // the second-K-stream kernels (pa_v2_decode_partial_extra): f16 / bf16 only
    return kv_dtype == PA_F16 || kv_dtype == PA_BF16 ? (group_size < 32 ? group_size : 32) : 0;
  if (head_dim != 64 && head_dim != 128) return 0;
  if (kv_dtype == PA_F16 || kv_dtype == PA_BF16) return group_size < 16 ? group_size : 16;
  if (kv_dtype == PA_F32) return group_size < 8 ? group_size : 8;
  return 0;
}

extern "C" pa_status pa_v2_default_target_ctas(int32_t device, int32_t num_qo_heads, int32_t num_kv_heads,
                                               int32_t head_dim, int32_t page_size, int32_t kv_dtype,
                                               int32_t* target_ctas) {
  if (!target_ctas || num_kv_heads < 1 || num_qo_heads < num_kv_heads || num_qo_heads % num_kv_heads ||
      page_size < 1)
    return PA_EINVAL;
  const int hpc = pa_v2_q_heads_per_cta(num_qo_heads / num_kv_heads, head_dim, kv_dtype);
  if (hpc == 0) return PA_EUNSUPPORTED;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return PA_ECUDA;
  if (device != prev && cudaSetDevice(device) != cudaSuccess) return PA_ECUDA;
  int sms = 0, per_sm = 0, rc = PA_ECUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) == cudaSuccess) {
    rc = head_dim == 512 ? pa::occupancy_partial_extra_tc05(kv_dtype, &per_sm)
         : pa::use_tensor_cores(kv_dtype, 0)
             ? pa::occupancy_partial_tc(kv_dtype, head_dim, hpc, pa::tc_uses_tma(page_size), &per_sm)
             : pa::occupancy_partial_simt(kv_dtype, head_dim, hpc, &per_sm);
  }
  if (device != prev) cudaSetDevice(prev);
  if (rc != PA_OK) return (pa_status)rc;
  if (per_sm < 1) return PA_ECUDA;
  *target_ctas = sms * per_sm;
  return PA_OK;
}

namespace {

struct FusedArgs {
  const int32_t* o_indptr;
  int32_t* counters;
  float* out;
  float* lse_final;
  const int32_t* member_rows;
  const int32_t* out_rows;
};

// Validate a decode launch and fill its launch arguments (tensor maps in *tm_k / *tm_v, which must outlive
// the launch); *tc / *tma say which kernel and staging it takes.  A plan with no chunks returns PA_OK with
// a->num_chunks = 0 and nothing to launch.
pa_status prepare_decode(const pa_v2_plan_t* plan, const float* q, const void* k_pool, const void* v_pool,
                         int32_t kv_dtype, int64_t num_pages, const int32_t* indices, int64_t num_indices,
                         const int32_t* indptr, const int32_t* last_page_len, const int32_t* first_page_offset,
                         const int32_t* request_indices, const int32_t* kv_tile_indices, float sm_scale,
                         float* v_out, float* lse2_out, int32_t* status, void* cuda_stream, const FusedArgs* fused,
                         pa::LaunchArgs* args, CUtensorMap* tm_k, CUtensorMap* tm_v, bool* tc_out, bool* tma_out) {
  if (!plan) return PA_EINVAL;
  args->num_chunks = 0;
  if (plan->num_chunks == 0) return PA_OK;
  if (!q || !k_pool || !v_pool || !indices || !indptr || !last_page_len || !first_page_offset ||
      !request_indices || !kv_tile_indices || !v_out || !lse2_out)
    return PA_EINVAL;
  if (fused && (!fused->o_indptr || !fused->counters || !fused->out || !fused->lse_final)) return PA_EINVAL;
  if (kv_dtype != plan->kv_dtype || num_pages < 1 || num_indices < plan->num_indices || plan->num_chunks < 0 ||
      plan->num_kv_heads < 1 || plan->q_groups < 1 || plan->page_size < 1 || !std::isfinite(sm_scale))
    return PA_EINVAL;
  if (!pa::aligned16(q) || !pa::aligned16(k_pool) || !pa::aligned16(v_pool) || !pa::aligned16(v_out) ||
      (fused && !pa::aligned16(fused->out)))
    return PA_EINVAL;
  const int D = plan->head_dim;
  const int ps = plan->page_size;
  if (D != 64 && D != 128) return PA_EUNSUPPORTED;  // head_dim 512 plans run pa_v2_decode_partial_extra
  if (num_pages * (int64_t)ps >= (1ll << 31)) return PA_EUNSUPPORTED;
  const int hpc = pa_v2_q_heads_per_cta(plan->num_qo_heads / plan->num_kv_heads, D, kv_dtype);
  if (hpc != plan->q_heads_per_cta) return PA_EINVAL;
  const int M = plan->stack_members;
  if (M < 1 || plan->out_row_step < 1) return PA_EINVAL;
  if (M > 1 && (plan->batch != 1 || plan->num_qo_heads % (M * plan->num_kv_heads) != 0)) return PA_EINVAL;
  const bool tc = pa::use_tensor_cores(kv_dtype, plan->kernel);
  if (!tc && hpc > 8) return PA_EUNSUPPORTED;
  const bool tma = !tc || pa::tc_uses_tma(ps);

  std::memset(tm_k, 0, sizeof(*tm_k));
  std::memset(tm_v, 0, sizeof(*tm_v));
  if (tma) {
    const int box_rows = ps <= pa::kStageRows ? ps : pa::kStageRows;
    const int box_d = tc ? 64 : D;
    const CUtensorMapSwizzle sw = tc ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE;
    if (!pa::make_pool_map(tm_k, k_pool, kv_dtype, num_pages * ps, plan->num_kv_heads, D, box_d, box_rows, sw) ||
        !pa::make_pool_map(tm_v, v_pool, kv_dtype, num_pages * ps, plan->num_kv_heads, D, box_d, box_rows, sw))
      return PA_ECUDA;
  }

  pa::LaunchArgs& a = *args;
  pa::PartialParams& p = a.p;
  std::memset(&p, 0, sizeof(p));
  p.q = q;
  p.indices = indices;
  p.indptr = indptr;
  p.last_page_len = last_page_len;
  p.first_page_offset = first_page_offset;
  p.request_indices = request_indices;
  p.kv_tile_indices = kv_tile_indices;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.v_out = v_out;
  p.lse_out = lse2_out;
  p.status = status;
  if (fused) {
    p.o_indptr = fused->o_indptr;
    p.counters = fused->counters;
    p.out = fused->out;
    p.lse_final = fused->lse_final;
    p.member_rows = fused->member_rows;
    p.out_rows = fused->out_rows;
    p.fused = 1;
  }
  p.num_pages = num_pages;
  p.num_indices = num_indices;
  // a one-request plan fixes chunk c to tile c of request 0 and that request's slots to 0 .. num_indices-1
  if (plan->batch == 1 && num_indices == plan->num_indices && num_indices > 0 && num_indices <= INT32_MAX)
    p.single_pages = (int32_t)num_indices;
  p.batch = plan->batch;
  p.num_qo_heads = plan->num_qo_heads;
  p.num_kv_heads = plan->num_kv_heads;
  p.group = plan->num_qo_heads / plan->num_kv_heads;
  p.hpc = hpc;
  p.q_groups = plan->q_groups;
  p.page_size = ps;
  p.pages_per_chunk = plan->pages_per_chunk;
  const pa::FastDiv fd = pa::FastDiv::make((uint32_t)ps);
  p.ps_magic = fd.magic;
  p.ps_shift = fd.shift;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.stack_members = M;
  p.member_heads = plan->num_qo_heads / M;
  p.member_group = p.group / M;
  p.out_row_step = plan->out_row_step;
  // The pre-wait L2 warm-up only for one-request plans, whose chunk geometry needs no load: their
  // speculative chain is one page-id load (~0.5 us when nothing runs before the kernel, against ~0.9 us
  // saved back to back, on GB300).  A batch's chain adds the chunk arrays and indptr ahead of the page
  // ids, which cost a one-step-at-a-time launch ~2 us for 0.35-0.5 us saved back to back.
  p.warm_l2 = p.single_pages > 0 ? 1 : 0;
  a.tm_k = tm_k;
  a.tm_v = tm_v;
  a.kv_dtype = kv_dtype;
  a.head_dim = D;
  a.num_chunks = plan->num_chunks;
  a.stream = static_cast<cudaStream_t>(cuda_stream);
  *tc_out = tc;
  *tma_out = tma;
  return PA_OK;
}

pa_status launch_decode(const pa_v2_plan_t* plan, const float* q, const void* k_pool, const void* v_pool,
                        int32_t kv_dtype, int64_t num_pages, const int32_t* indices, int64_t num_indices,
                        const int32_t* indptr, const int32_t* last_page_len, const int32_t* first_page_offset,
                        const int32_t* request_indices, const int32_t* kv_tile_indices, float sm_scale,
                        float* v_out, float* lse2_out, int32_t* status, void* cuda_stream, const FusedArgs* fused,
                        bool warm_l2 = true) {
  alignas(64) CUtensorMap tm_k, tm_v;
  pa::LaunchArgs a;
  bool tc = false, tma = false;
  const pa_status rc = prepare_decode(plan, q, k_pool, v_pool, kv_dtype, num_pages, indices, num_indices, indptr,
                                      last_page_len, first_page_offset, request_indices, kv_tile_indices, sm_scale,
                                      v_out, lse2_out, status, cuda_stream, fused, &a, &tm_k, &tm_v, &tc, &tma);
  if (rc != PA_OK || a.num_chunks == 0) return rc;
  if (!warm_l2) a.p.warm_l2 = 0;
  return (pa_status)(tc ? pa::launch_partial_tc(a, tma) : pa::launch_partial_simt(a));
}

}  // namespace

extern "C" pa_status pa_v2_decode_partial(const pa_v2_plan_t* plan, const float* q, const void* k_pool,
                                          const void* v_pool, int32_t kv_dtype, int64_t num_pages,
                                          const int32_t* indices, int64_t num_indices, const int32_t* indptr,
                                          const int32_t* last_page_len, const int32_t* first_page_offset,
                                          const int32_t* request_indices, const int32_t* kv_tile_indices,
                                          float sm_scale, float* v_out, float* lse2_out, int32_t* status,
                                          void* cuda_stream) {
  return launch_decode(plan, q, k_pool, v_pool, kv_dtype, num_pages, indices, num_indices, indptr, last_page_len,
                       first_page_offset, request_indices, kv_tile_indices, sm_scale, v_out, lse2_out, status,
                       cuda_stream, nullptr);
}

namespace pa {

pa_status decode_partial_leading(const pa_v2_plan_t* plan, const float* q, const void* k_pool, const void* v_pool,
                                 int32_t kv_dtype, int64_t num_pages, const int32_t* indices, int64_t num_indices,
                                 const int32_t* indptr, const int32_t* last_page_len,
                                 const int32_t* first_page_offset, const int32_t* request_indices,
                                 const int32_t* kv_tile_indices, float sm_scale, float* v_out, float* lse2_out,
                                 int32_t* status, void* cuda_stream) {
  return launch_decode(plan, q, k_pool, v_pool, kv_dtype, num_pages, indices, num_indices, indptr, last_page_len,
                       first_page_offset, request_indices, kv_tile_indices, sm_scale, v_out, lse2_out, status,
                       cuda_stream, nullptr, false);
}

}  // namespace pa

extern "C" pa_status pa_v2_decode(const pa_v2_plan_t* plan, const float* q, const void* k_pool, const void* v_pool,
                                  int32_t kv_dtype, int64_t num_pages, const int32_t* indices, int64_t num_indices,
                                  const int32_t* indptr, const int32_t* last_page_len,
                                  const int32_t* first_page_offset, const int32_t* request_indices,
                                  const int32_t* kv_tile_indices, const int32_t* o_indptr, float sm_scale,
                                  float* workspace_v, float* workspace_lse, int32_t* counters, float* out,
                                  float* lse2_out, const int32_t* member_rows, const int32_t* out_rows,
                                  int32_t* status, void* cuda_stream) {
  const FusedArgs f{o_indptr, counters, out, lse2_out, member_rows, out_rows};
  return launch_decode(plan, q, k_pool, v_pool, kv_dtype, num_pages, indices, num_indices, indptr, last_page_len,
                       first_page_offset, request_indices, kv_tile_indices, sm_scale, workspace_v, workspace_lse,
                       status, cuda_stream, &f);
}

// Both cascade levels in one launch of the tensor-core kernel, writing every chunk's partial into the rows
// of one merge input, then the merge of each request's rows (cascade-attention.md, composition paragraphs).
extern "C" pa_status pa_v2_cascade_decode(const pa_v2_plan_t* plan0, const pa_v2_plan_t* plan1,
                                          const pa_v2_cascade_level_t* level0, const pa_v2_cascade_level_t* level1,
                                          const float* q, const void* k_pool, const void* v_pool, int32_t kv_dtype,
                                          int64_t num_pages, float sm_scale, float* merge_v, float* merge_lse,
                                          int32_t merge_rows, const int32_t* merge_indptr, int32_t batch_out,
                                          float* out, float* lse2_out, int32_t* status, void* cuda_stream) {
  if (!plan0 || !plan1 || !level0 || !level1 || !merge_v || !merge_lse || !merge_indptr || !out || !lse2_out ||
      merge_rows < 0 || batch_out < 0 || !level0->part_rows || (plan1->num_chunks > 0 && !level1->part_rows))
    return PA_EINVAL;
  if (plan0->stack_members < 1 || plan0->kv_dtype != plan1->kv_dtype || plan0->head_dim != plan1->head_dim ||
      plan0->page_size != plan1->page_size || plan0->num_kv_heads != plan1->num_kv_heads ||
      plan0->num_qo_heads != plan1->num_qo_heads * plan0->stack_members || plan1->stack_members != 1)
    return PA_EUNSUPPORTED;
  const pa_v2_cascade_level_t* lv[2] = {level0, level1};
  const pa_v2_plan_t* pl[2] = {plan0, plan1};
  alignas(64) CUtensorMap tk[2], tv[2];
  pa::LaunchArgs a[2];
  bool tc[2] = {false, false}, tma[2] = {false, false};
  for (int l = 0; l < 2; ++l) {
    const pa_status rc =
        prepare_decode(pl[l], q, k_pool, v_pool, kv_dtype, num_pages, lv[l]->indices, lv[l]->num_indices,
                       lv[l]->indptr, lv[l]->last_page_len, lv[l]->first_page_offset, lv[l]->request_indices,
                       lv[l]->kv_tile_indices, sm_scale, merge_v, merge_lse, status, cuda_stream, nullptr, &a[l],
                       &tk[l], &tv[l], &tc[l], &tma[l]);
    if (rc != PA_OK) return rc;
    a[l].p.part_rows = lv[l]->part_rows;
    a[l].p.part_limit = (int64_t)merge_rows * plan1->num_qo_heads;
    a[l].p.member_rows = lv[l]->member_rows;
  }
  if (a[0].num_chunks == 0 || a[1].num_chunks == 0) return PA_EINVAL;  // each level has at least one chunk
  if (!tc[0] || !tc[1] || tma[0] != tma[1]) return PA_EUNSUPPORTED;
  // one launch: the tensor maps depend only on the shared pools, dtype, page size and head counts
  const int rc = pa::launch_partial_tc_two_plans(a[0], a[1].p, a[1].num_chunks, tma[0]);
  if (rc != PA_OK) return (pa_status)rc;
  return pa_merge_states(merge_v, merge_lse, merge_indptr, batch_out, merge_rows, plan1->num_qo_heads,
                         plan1->head_dim, out, lse2_out, status, cuda_stream);
}
