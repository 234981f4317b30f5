// pa_merge.cu -- the variable-length merge-state kernel and its C-ABI launcher.
//
// Issue #898 ("Fused paged-attention decode v2: CSR page table, cross-CTA
// split-KV, and variable-length merge kernels"), design piece 3, and PR #984
// ("fused paged-attention decode v2 with CSR page table and cross-CTA
// split-KV"), What changed 3: partial attention states (v_i, lse_i), each v_i
// already normalized and lse_i in log2 units, combine by
//   m = max lse_i, w_i = 2^(lse_i - m), v = sum w_i v_i / sum w_i,
//   lse = log2(sum w_i) + m
// over the rows o_indptr[r] .. o_indptr[r+1]-1 of output row r.  -inf rows
// weigh 0; a group without a finite row yields zeros and -inf.  One row is an
// exact identity (w = 1).
//
// Layout on sm_103a: the merge reads little data (the partial workspace) and
// is bound by memory latency, so it is organised to need one round of loads
// for up to 32 partial rows.  One CTA of 4 warps per (output row, head): warp w
// loads the LSE and the 128-bit V slice (4 head-dim floats per lane) of rows
// i0 + w, i0 + w + 4, ... eight at a time, keeps a running maximum and rescales
// its sum when the maximum grows, and the four warps' (max, weight sum, V sum)
// meet in shared memory, each scaled by 2^(its max - the group max).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "pa_device.cuh"
#include "pa_launch.h"
#include "pa_v2.h"

namespace pa {
namespace {

constexpr int kMergeWarps = 4;
constexpr int kMergeUnroll = 8;

__device__ __forceinline__ float merge_weight(float l, float m) {
  return l == -INFINITY ? 0.f : fast_exp2(l - m);
}

// NV > 0: head_dim % 4 == 0 and head_dim <= 128 * NV (NV float4 per lane:
// 1 up to head_dim 128, 4 up to 512); NV == 0: a scalar loop over head_dim.
template <int NV>
__device__ __forceinline__ void merge_body(const float* __restrict__ v_in, const float* __restrict__ lse_in,
                                           const int32_t* __restrict__ o_indptr, int32_t num_rows_out,
                                           int32_t num_partials, int32_t num_heads, int32_t head_dim,
                                           float* __restrict__ v_out, float* __restrict__ lse_out,
                                           int32_t* status) {
  __shared__ float red[kMergeWarps];
  __shared__ float wsum_s[kMergeWarps];
  constexpr bool VECTOR = NV > 0;
  constexpr int U = NV > 1 ? kMergeUnroll / 2 : kMergeUnroll;  // rows in flight per warp
  __shared__ __align__(16) float acc_s[kMergeWarps][VECTOR ? 128 * NV : 4];

  // the kernel that follows (normally the next step's partial kernel) may be
  // scheduled now; it waits for this grid to finish
  pdl_launch_dependents();
  // launched as a programmatic dependent of the partial kernel: wait for its
  // grid to complete (and its writes to be visible) before reading anything
  pdl_wait_prerequisites();

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x / num_heads;
  const int h = blockIdx.x % num_heads;
  int i0 = o_indptr[r];
  int i1 = o_indptr[r + 1];
  if (i0 < 0 || i1 < i0 || i1 > num_partials) {
    if (threadIdx.x == 0) report(status, PA_DEVICE_BAD_INDPTR);
    i0 = i1 = 0;
  }
  const size_t hs = (size_t)num_heads;

  float* out = v_out + ((size_t)r * num_heads + h) * head_dim;
  if (VECTOR) {
    const int d4n = head_dim >> 2;
    float m = -INFINITY, ws = 0.f;
    float4 acc[NV > 0 ? NV : 1];
#pragma unroll
    for (int k = 0; k < NV; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = i0 + warp; base < i1; base += kMergeWarps * U) {
      float l[U];
      float4 v[U][NV > 0 ? NV : 1];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = base + u * kMergeWarps;
        l[u] = i < i1 ? lse_in[i * hs + h] : -INFINITY;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
          const int q4 = lane + 32 * k;
          v[u][k] = (i < i1 && q4 < d4n) ? reinterpret_cast<const float4*>(v_in + (i * hs + h) * head_dim)[q4]
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float mb = m;
#pragma unroll
      for (int u = 0; u < U; ++u) mb = fmaxf(mb, l[u]);
      if (mb == -INFINITY) continue;
      const float sc = merge_weight(m, mb);  // 0 while nothing has been summed
      ws *= sc;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        acc[k].x *= sc;
        acc[k].y *= sc;
        acc[k].z *= sc;
        acc[k].w *= sc;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float w = merge_weight(l[u], mb);
        ws += w;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
          acc[k].x = fmaf(w, v[u][k].x, acc[k].x);
          acc[k].y = fmaf(w, v[u][k].y, acc[k].y);
          acc[k].z = fmaf(w, v[u][k].z, acc[k].z);
          acc[k].w = fmaf(w, v[u][k].w, acc[k].w);
        }
      }
      m = mb;
    }
#pragma unroll
    for (int k = 0; k < NV; ++k)
      if (lane + 32 * k < d4n) reinterpret_cast<float4*>(acc_s[warp])[lane + 32 * k] = acc[k];
    if (lane == 0) {
      red[warp] = m;
      wsum_s[warp] = ws;
    }
    __syncwarp();  // reconverge the per-lane branches before the aligned barrier
    __syncthreads();
    float M = red[0];
#pragma unroll
    for (int w = 1; w < kMergeWarps; ++w) M = fmaxf(M, red[w]);
    if (M == -INFINITY) {
      for (int d = threadIdx.x; d < head_dim; d += kMergeWarps * 32) out[d] = 0.f;
      if (threadIdx.x == 0) lse_out[(size_t)r * num_heads + h] = -INFINITY;
      return;
    }
    float scw[kMergeWarps];
    float W = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) {
      scw[w] = merge_weight(red[w], M);
      W = fmaf(wsum_s[w], scw[w], W);
    }
    for (int d = threadIdx.x; d < head_dim; d += kMergeWarps * 32) {
      float a = 0.f;
#pragma unroll
      for (int w = 0; w < kMergeWarps; ++w) a = fmaf(acc_s[w][d], scw[w], a);
      out[d] = a / W;
    }
    if (threadIdx.x == 0) lse_out[(size_t)r * num_heads + h] = fast_log2(W) + M;
  } else {
    // general head_dim: the whole CTA walks the rows, one head-dim element per thread
    float m = -INFINITY;
    for (int i = i0 + threadIdx.x; i < i1; i += kMergeWarps * 32) m = fmaxf(m, lse_in[i * hs + h]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncwarp();
    __syncthreads();
    m = red[0];
#pragma unroll
    for (int w = 1; w < kMergeWarps; ++w) m = fmaxf(m, red[w]);
    if (m == -INFINITY) {
      for (int d = threadIdx.x; d < head_dim; d += kMergeWarps * 32) out[d] = 0.f;
      if (threadIdx.x == 0) lse_out[(size_t)r * num_heads + h] = -INFINITY;
      return;
    }
    float W = 0.f;
    for (int i = i0; i < i1; ++i) W += merge_weight(lse_in[i * hs + h], m);
    for (int d = threadIdx.x; d < head_dim; d += kMergeWarps * 32) {
      float a = 0.f;
      for (int i = i0; i < i1; ++i) a = fmaf(merge_weight(lse_in[i * hs + h], m), v_in[(i * hs + h) * head_dim + d], a);
      out[d] = a / W;
    }
    if (threadIdx.x == 0) lse_out[(size_t)r * num_heads + h] = fast_log2(W) + m;
  }
}

// done (or null): a counter in memory the host can read; each CTA adds one once
// its results are visible system-wide, so a host thread can wait for the count
// instead of synchronising the stream.
template <int NV>
__global__ void __launch_bounds__(kMergeWarps * 32)
    pa_merge_states_kernel(const float* __restrict__ v_in, const float* __restrict__ lse_in,
                           const int32_t* __restrict__ o_indptr, int32_t num_rows_out, int32_t num_partials,
                           int32_t num_heads, int32_t head_dim, float* __restrict__ v_out,
                           float* __restrict__ lse_out, int32_t* status, int32_t* done) {
  merge_body<NV>(v_in, lse_in, o_indptr, num_rows_out, num_partials, num_heads, head_dim, v_out, lse_out, status);
  if (done) {
    __threadfence_system();  // this thread's results (and status bits) before the count
    __syncthreads();
    if (threadIdx.x == 0) atomicAdd_system(done, 1);
  }
}

}  // namespace

pa_status launch_merge(const float* v_in, const float* lse2_in, const int32_t* o_indptr, int32_t num_rows_out,
                       int32_t num_partials, int32_t num_heads, int32_t head_dim, float* v_out, float* lse2_out,
                       int32_t* status, int32_t* done, int64_t* ctas, void* cuda_stream) {
  if (num_rows_out < 0 || num_partials < 0 || num_heads < 1 || head_dim < 1) return PA_EINVAL;
  if (ctas) *ctas = 0;
  if (num_rows_out == 0) return PA_OK;
  if (!o_indptr || !v_out || !lse2_out || (num_partials > 0 && (!v_in || !lse2_in))) return PA_EINVAL;
  const int nv = head_dim % 4 != 0 ? 0 : head_dim <= 128 ? 1 : head_dim <= 512 ? 4 : 0;
  const bool vec = nv > 0;
  if (vec && (((uintptr_t)v_in | (uintptr_t)v_out) & 15u)) return PA_EINVAL;
  const long long blocks = (long long)num_rows_out * num_heads;
  if (blocks > 0x7fffffffLL) return PA_EUNSUPPORTED;
  // Programmatic dependent launch: the merge may be scheduled while the kernel
  // before it in the stream (normally the partial kernel) is still running; the
  // kernel's first instruction waits for that grid to complete.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(cuda_stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  auto fn = nv == 1 ? pa_merge_states_kernel<1> : nv == 4 ? pa_merge_states_kernel<4> : pa_merge_states_kernel<0>;
  cudaError_t rc = cudaLaunchKernelEx(&cfg, fn, v_in, lse2_in, o_indptr, num_rows_out, num_partials, num_heads,
                                      head_dim, v_out, lse2_out, status, done);
  if (rc != cudaSuccess || cudaGetLastError() != cudaSuccess) return PA_ECUDA;
  if (ctas) *ctas = blocks;
  return PA_OK;
}

}  // namespace pa

extern "C" pa_status pa_merge_states(const float* v_in, const float* lse2_in, const int32_t* o_indptr,
                                     int32_t num_rows_out, int32_t num_partials, int32_t num_heads,
                                     int32_t head_dim, float* v_out, float* lse2_out, int32_t* status,
                                     void* cuda_stream) {
  return pa::launch_merge(v_in, lse2_in, o_indptr, num_rows_out, num_partials, num_heads, head_dim, v_out, lse2_out,
                          status, nullptr, nullptr, cuda_stream);
}
