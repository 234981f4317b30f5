// pa_partial_extra.cu -- split-KV partial kernel with a second K stream
// (MLA / DSA decode), CUDA cores.
//
// sparse-paged-decode.md (issue #904), the DSA paragraphs, third way out: the
// score of token t is
//   scale * (q . k[row_t][0:Dim]) + scale * (q_extra . k_extra[row_t][0:ExtraDim])
// and the output averages v[row_t][0:Dim].  K rows sit in an allocation whose
// row stride (RowStride) may exceed Dim -- the DSA K buffer is
// concat(kv_latent, indexer_key) with Dim = kv_lora_rank -- and k_extra is a
// second allocation (k_pe, ExtraDim = qk_rope_head_dim) that shares the row
// mapping.  In MLA the values are the latent rows themselves (v_pool is the K
// allocation) and the kernel reuses the key registers as values.  Rows resolve
// through the same CSR page table as the single-stream decode: chunk = run of
// page slots, token i of request r at indices[indptr[r] + (fpo + i) / ps],
// entry (fpo + i) % ps; one CTA per (chunk, kv head, q-head group).
//
// Shapes served: Dim 512, ExtraDim 64 (DeepSeek's kv_lora_rank and
// qk_rope_head_dim), 8 query heads per CTA, f16 / bf16 pools.  This file also
// holds the entry point, which picks the kernel by plan.kernel: 0 the
// tensor-memory kernel (pa_partial_extra_tc05.cu) when the values are the key
// rows, else the warp-level tensor-core kernel (pa_partial_extra_tc.cu, also
// plan.kernel 2); 1 this CUDA-core kernel.  The plans group up to 32 query
// heads per CTA; the 8-head kernels regroup them at launch.
//
// Layout: 4 warps, each owning 2 of the CTA's query heads; all four read the
// same K / V rows (the later ones from L1).  Lane l owns latent dims
// 16l .. 16l+15 (two 16-byte loads per row) and extra dims 2l, 2l+1, with the
// matching query values (f32, scale * log2(e) folded in) in registers.  Two
// tokens are scored per iteration (independent loads and shuffle trees), the
// dot products reduced across lanes with butterfly shuffles, the online
// softmax kept in f32 in every lane, and the output accumulated in the lane's
// 16 dims x 2 heads.  No shared memory, no barriers.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int kXDim = 512;        // Dim
constexpr int kXExtra = 64;       // ExtraDim
constexpr int kXWarps = 4;
constexpr int kXHeadsPerWarp = 2;
constexpr int kXHeads = kXWarps * kXHeadsPerWarp;  // 8 query heads per CTA
constexpr int kXTok = 2;          // tokens per iteration
constexpr int kXLaneDims = kXDim / 32;             // 16 latent dims per lane
constexpr int kXLaneExtra = kXExtra / 32;          // 2 extra dims per lane

struct ExtraFields {
  const float* q_extra;  // [B, Hq, ExtraDim]
  const void* k_extra;   // extra rows
  int64_t k_stride;      // elements between consecutive (row, kv head) entries of each allocation
  int64_t v_stride;
  int64_t e_stride;
};

template <typename T> struct XT;
template <> struct XT<__half> {
  __device__ __forceinline__ static float2 f2(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  }
};
template <> struct XT<__nv_bfloat16> {
  __device__ __forceinline__ static float2 f2(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  }
};

template <typename T, bool SHARED_V>
__global__ void __launch_bounds__(kXWarps * 32, 4)
    pa_v2_partial_extra_kernel(const PartialParams p, const ExtraFields x) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
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
  // visible tokens of this chunk: [t0, t1)
  const int seq = gm.pages > 0 ? (gm.pages - 1) * ps + gm.lpl - gm.fpo : 0;
  const int t0 = gm.n_stages > 0 ? max(0, gm.s_begin * ps - gm.fpo) : 0;
  const int t1 = gm.n_stages > 0 ? min(seq, gm.s_end * ps - gm.fpo) : 0;

  // this warp's heads and their query values for the lane's dims
  float qd[kXHeadsPerWarp][kXLaneDims], qe[kXHeadsPerWarp][kXLaneExtra];
#pragma unroll
  for (int h = 0; h < kXHeadsPerWarp; ++h) {
    const int head = warp * kXHeadsPerWarp + h;
    const bool hv = head < nheads;
    const size_t qrow = (size_t)r * p.num_qo_heads + h_first + (hv ? head : 0);
    const float4* qv = reinterpret_cast<const float4*>(p.q + qrow * kXDim + lane * kXLaneDims);
#pragma unroll
    for (int i = 0; i < kXLaneDims / 4; ++i) {
      const float4 v = hv ? qv[i] : make_float4(0.f, 0.f, 0.f, 0.f);
      qd[h][4 * i + 0] = v.x * p.scale_log2;
      qd[h][4 * i + 1] = v.y * p.scale_log2;
      qd[h][4 * i + 2] = v.z * p.scale_log2;
      qd[h][4 * i + 3] = v.w * p.scale_log2;
    }
    const float2 e = hv ? *reinterpret_cast<const float2*>(x.q_extra + qrow * kXExtra + lane * kXLaneExtra)
                        : make_float2(0.f, 0.f);
    qe[h][0] = e.x * p.scale_log2;
    qe[h][1] = e.y * p.scale_log2;
  }

  float m_run[kXHeadsPerWarp], l_run[kXHeadsPerWarp], o[kXHeadsPerWarp][kXLaneDims];
#pragma unroll
  for (int h = 0; h < kXHeadsPerWarp; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.f;
#pragma unroll
    for (int d = 0; d < kXLaneDims; ++d) o[h][d] = 0.f;
  }

  const T* kpool = static_cast<const T*>(p.k_pool);
  const T* vpool = static_cast<const T*>(p.v_pool);
  const T* epool = static_cast<const T*>(x.k_extra);

  for (int t = t0; t < t1; t += kXTok) {
    uint4 kw[kXTok][2], vw[kXTok][2];
    uint32_t ew[kXTok];
    bool valid[kXTok];
#pragma unroll
    for (int u = 0; u < kXTok; ++u) {
      const int tok = t + u;
      valid[u] = false;
      kw[u][0] = kw[u][1] = vw[u][0] = vw[u][1] = make_uint4(0u, 0u, 0u, 0u);
      ew[u] = 0u;
      if (tok < t1) {
        const int pos = gm.fpo + tok;
        const int slot = (int)fast_div((uint32_t)pos, p.ps_magic, p.ps_shift);
        const int e = pos - slot * ps;
        const int32_t page = __ldg(p.indices + gm.slot_base + slot);
        if (page >= 0 && (int64_t)page < p.num_pages) {
          valid[u] = true;
          const int64_t row = ((int64_t)page * ps + e) * p.num_kv_heads + kvh;
          const uint4* kr = reinterpret_cast<const uint4*>(kpool + row * x.k_stride + lane * kXLaneDims);
          kw[u][0] = __ldg(kr);
          kw[u][1] = __ldg(kr + 1);
          if (!SHARED_V) {
            const uint4* vr = reinterpret_cast<const uint4*>(vpool + row * x.v_stride + lane * kXLaneDims);
            vw[u][0] = __ldg(vr);
            vw[u][1] = __ldg(vr + 1);
          }
          ew[u] = __ldg(reinterpret_cast<const uint32_t*>(epool + row * x.e_stride + lane * kXLaneExtra));
        } else if (lane == 0) {
          report(p.status, PA_DEVICE_BAD_PAGE);
        }
      }
    }

    // scores: lane partials, then a butterfly over the warp
    float s[kXTok][kXHeadsPerWarp];
#pragma unroll
    for (int u = 0; u < kXTok; ++u) {
      float kf[kXLaneDims];
      const uint32_t* w = reinterpret_cast<const uint32_t*>(&kw[u][0]);
#pragma unroll
      for (int i = 0; i < kXLaneDims / 2; ++i) {
        const float2 f = XT<T>::f2(w[i]);
        kf[2 * i] = f.x;
        kf[2 * i + 1] = f.y;
      }
      const float2 ef = XT<T>::f2(ew[u]);
#pragma unroll
      for (int h = 0; h < kXHeadsPerWarp; ++h) {
        float a0 = qe[h][0] * ef.x, a1 = qe[h][1] * ef.y;
#pragma unroll
        for (int d = 0; d < kXLaneDims; d += 2) {
          a0 = fmaf(qd[h][d], kf[d], a0);
          a1 = fmaf(qd[h][d + 1], kf[d + 1], a1);
        }
        s[u][h] = a0 + a1;
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
      for (int u = 0; u < kXTok; ++u)
#pragma unroll
        for (int h = 0; h < kXHeadsPerWarp; ++h) s[u][h] += __shfl_xor_sync(0xffffffffu, s[u][h], off);

    // online softmax over the kXTok tokens, per head
    float pw[kXTok][kXHeadsPerWarp];
#pragma unroll
    for (int h = 0; h < kXHeadsPerWarp; ++h) {
      float mx = -INFINITY;
#pragma unroll
      for (int u = 0; u < kXTok; ++u) {
        if (!valid[u]) s[u][h] = -INFINITY;
        mx = fmaxf(mx, s[u][h]);
      }
      const float mn = fmaxf(m_run[h], mx);
      const float mu = mn == -INFINITY ? 0.f : mn;
      const float alpha = fast_exp2(m_run[h] - mu);
      m_run[h] = mn;
      float sum = 0.f;
#pragma unroll
      for (int u = 0; u < kXTok; ++u) {
        pw[u][h] = fast_exp2(s[u][h] - mu);
        sum += pw[u][h];
      }
      l_run[h] = l_run[h] * alpha + sum;
#pragma unroll
      for (int d = 0; d < kXLaneDims; ++d) o[h][d] *= alpha;
    }

    // o += p . v (the lane's 16 dims)
#pragma unroll
    for (int u = 0; u < kXTok; ++u) {
      const uint32_t* w = reinterpret_cast<const uint32_t*>(SHARED_V ? &kw[u][0] : &vw[u][0]);
#pragma unroll
      for (int i = 0; i < kXLaneDims / 2; ++i) {
        const float2 f = XT<T>::f2(w[i]);
#pragma unroll
        for (int h = 0; h < kXHeadsPerWarp; ++h) {
          o[h][2 * i] = fmaf(pw[u][h], f.x, o[h][2 * i]);
          o[h][2 * i + 1] = fmaf(pw[u][h], f.y, o[h][2 * i + 1]);
        }
      }
    }
  }

  // normalized partial and lse2 of this chunk for the warp's heads
  const size_t hq = (size_t)p.num_qo_heads;
#pragma unroll
  for (int h = 0; h < kXHeadsPerWarp; ++h) {
    const int head = warp * kXHeadsPerWarp + h;
    if (head >= nheads) continue;
    const float inv = l_run[h] > 0.f ? 1.f / l_run[h] : 0.f;
    float4* dst = reinterpret_cast<float4*>(p.v_out + ((size_t)c * hq + h_first + head) * kXDim + lane * kXLaneDims);
#pragma unroll
    for (int i = 0; i < kXLaneDims / 4; ++i)
      dst[i] = make_float4(o[h][4 * i] * inv, o[h][4 * i + 1] * inv, o[h][4 * i + 2] * inv, o[h][4 * i + 3] * inv);
    if (lane == 0)
      p.lse_out[(size_t)c * hq + h_first + head] = l_run[h] > 0.f ? m_run[h] + fast_log2(l_run[h]) : -INFINITY;
  }
}

struct ExtraInstance {
  void (*fn)(const PartialParams, const ExtraFields);
};

bool extra_pick(int kv_dtype, bool shared_v, ExtraInstance* out) {
  if (kv_dtype == PA_F16) {
    out->fn = shared_v ? pa_v2_partial_extra_kernel<__half, true> : pa_v2_partial_extra_kernel<__half, false>;
    return true;
  }
  if (kv_dtype == PA_BF16) {
    out->fn = shared_v ? pa_v2_partial_extra_kernel<__nv_bfloat16, true>
                       : pa_v2_partial_extra_kernel<__nv_bfloat16, false>;
    return true;
  }
  return false;
}

}  // namespace

int occupancy_partial_extra(int kv_dtype, int* blocks_per_sm) {
  ExtraInstance inst;
  if (!extra_pick(kv_dtype, true, &inst)) return PA_EUNSUPPORTED;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, inst.fn, kXWarps * 32, 0) == cudaSuccess
             ? PA_OK
             : PA_ECUDA;
}

}  // namespace pa

namespace {

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

}  // namespace

extern "C" pa_status pa_v2_decode_partial_extra(
    const pa_v2_plan_t* plan, const float* q, const float* q_extra, const void* k_pool, int64_t k_row_stride,
    const void* v_pool, int64_t v_row_stride, const void* k_extra_pool, int64_t k_extra_row_stride,
    int32_t extra_dim, int32_t kv_dtype, int64_t num_pages, const int32_t* indices, int64_t num_indices,
    const int32_t* indptr, const int32_t* last_page_len, const int32_t* first_page_offset,
    const int32_t* request_indices, const int32_t* kv_tile_indices, float sm_scale, float* v_out,
    float* lse2_out, int32_t* status, void* cuda_stream) {
  using namespace pa;
  if (!plan || plan->head_dim != kXDim || extra_dim != kXExtra) return PA_EUNSUPPORTED;
  if (kv_dtype != plan->kv_dtype || (kv_dtype != PA_F16 && kv_dtype != PA_BF16)) return PA_EUNSUPPORTED;
  if (plan->num_chunks < 0 || plan->batch < 0 || num_pages < 1 || num_indices < plan->num_indices ||
      !std::isfinite(sm_scale))
    return PA_EINVAL;
  if (plan->num_chunks == 0) return PA_OK;
  if (!q || !q_extra || !k_pool || !v_pool || !k_extra_pool || !indices || !indptr || !last_page_len ||
      !first_page_offset || !request_indices || !kv_tile_indices || !v_out || !lse2_out)
    return PA_EINVAL;
  const int G = plan->num_qo_heads / plan->num_kv_heads;
  if (plan->q_heads_per_cta != pa_v2_q_heads_per_cta(G, kXDim, kv_dtype) || plan->stack_members != 1 ||
      plan->out_row_step != 1 || plan->kernel < 0 || plan->kernel > 2)
    return PA_EINVAL;
  // rows are read 16 bytes (extra rows 4 bytes) at a time from 16-byte-aligned row starts;
  // q and v_out are read / written as float4 and q_extra as float2
  if (k_row_stride < kXDim || v_row_stride < kXDim || k_extra_row_stride < kXExtra || k_row_stride % 8 ||
      v_row_stride % 8 || k_extra_row_stride % 8 || !aligned16(k_pool) || !aligned16(v_pool) ||
      !aligned16(k_extra_pool) || !aligned16(q) || !aligned16(v_out) ||
      (reinterpret_cast<uintptr_t>(q_extra) & 7u))
    return PA_EINVAL;
  if (num_pages * plan->page_size >= (1ll << 31)) return PA_EUNSUPPORTED;
  const bool shared_v = v_pool == k_pool && v_row_stride == k_row_stride;
  ExtraInstance inst;
  if (!extra_pick(kv_dtype, shared_v, &inst)) return PA_EUNSUPPORTED;
  // plan->kernel 0: the tensor-memory kernel (values in the key tile) or, for separate values, the
  // warp-level tensor-core kernel; 1: CUDA cores; 2: the warp-level tensor-core kernel
  const bool tc05 = plan->kernel == 0 && shared_v;
  const bool tc = plan->kernel != 1;

  PartialParams p;
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
  p.stack_members = 1;
  p.out_row_step = 1;
  p.num_pages = num_pages;
  p.num_indices = num_indices;
  // a one-request plan fixes chunk c to tile c of request 0 and that request's slots to 0 .. num_indices-1
  if (plan->batch == 1 && num_indices == plan->num_indices && num_indices > 0 && num_indices <= INT32_MAX)
    p.single_pages = (int32_t)num_indices;
  p.batch = plan->batch;
  p.num_qo_heads = plan->num_qo_heads;
  p.num_kv_heads = plan->num_kv_heads;
  p.group = G;
  p.hpc = plan->q_heads_per_cta;
  p.q_groups = plan->q_groups;
  if (!tc05) {  // the other kernels serve 8 query heads per CTA: regroup the plan's heads
    p.hpc = G < kXHeads ? G : kXHeads;
    p.q_groups = (G + p.hpc - 1) / p.hpc;
  }
  p.page_size = plan->page_size;
  p.pages_per_chunk = plan->pages_per_chunk;
  const FastDiv fd = FastDiv::make((uint32_t)plan->page_size);
  p.ps_magic = fd.magic;
  p.ps_shift = fd.shift;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  ExtraFields x;
  x.q_extra = q_extra;
  x.k_extra = k_extra_pool;
  x.k_stride = k_row_stride;
  x.v_stride = v_row_stride;
  x.e_stride = k_extra_row_stride;

  const dim3 grid((unsigned)plan->num_chunks, (unsigned)(plan->num_kv_heads * p.q_groups));
  if (tc05)
    return (pa_status)launch_partial_extra_tc05(p, q_extra, k_extra_pool, k_row_stride, k_extra_row_stride,
                                                kv_dtype, grid, static_cast<cudaStream_t>(cuda_stream));
  if (tc)
    return (pa_status)launch_partial_extra_tc(p, q_extra, k_extra_pool, k_row_stride, v_row_stride,
                                              k_extra_row_stride, shared_v, kv_dtype, grid,
                                              static_cast<cudaStream_t>(cuda_stream));
  const cudaError_t rc =
      launch_dependent(inst.fn, grid, dim3(kXWarps * 32), 0, static_cast<cudaStream_t>(cuda_stream), p, x);
  return rc == cudaSuccess && cudaGetLastError() == cudaSuccess ? PA_OK : PA_ECUDA;
}
