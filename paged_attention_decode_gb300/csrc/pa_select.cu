// pa_select.cu -- block -> token expansion of a block-sparse selection, and
// the host-side CSR structure of the resulting token-exact page table.
//
// sparse-paged-decode.md (issue #904): a model that selects blocks of
// positions still reaches a token-exact (page_size 1) page table by expanding
// the selected block ids into token rows in one pass over the selected rows;
// the final block, the query's own, is appended unconditionally with its live
// rows only, which keeps the per-request row count a function of kv_len and
// keeps every row inside the live window.  The row count is host data, so the
// CSR structure (indptr, last_page_len, first_page_offset) is built on the
// host from (requests, rows per request) alone and nothing is read back.
//
// One thread per output row: the writes are coalesced, the block id of a row
// is a broadcast load shared by block_size consecutive threads.  The pass
// moves 4 bytes per selected row, against 2 * D * esize bytes of K/V the
// decode then reads for it.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "pa_device.cuh"
#include "pa_internal.cuh"
#include "pa_v2.h"

namespace pa {
namespace {

constexpr int kSelectThreads = 256;

__global__ void __launch_bounds__(kSelectThreads)
    pa_selection_from_blocks_kernel(const int32_t* __restrict__ block_ids, int32_t topk, int32_t block_size,
                                    int32_t num_blocks, int32_t per_request, int32_t total, int64_t request_stride,
                                    int32_t* __restrict__ indices, int32_t* status) {
  pdl_launch_dependents();
  pdl_wait_prerequisites();
  const int64_t stride = (int64_t)gridDim.x * kSelectThreads;
  for (int64_t o64 = (int64_t)blockIdx.x * kSelectThreads + threadIdx.x; o64 < total; o64 += stride) {
    const int32_t o = (int32_t)o64;  // total <= INT32_MAX
    const int32_t r = o / per_request;
    const int32_t w = o - r * per_request;
    const int32_t slot = w / block_size;
    const int32_t e = w - slot * block_size;
    int32_t block = num_blocks - 1;  // past the selected slots: the final block
    if (slot < topk) {
      block = __ldg(block_ids + (int64_t)r * topk + slot);
      if (block < 0 || block >= num_blocks - 1) {
        if (e == 0) report(status, PA_DEVICE_BAD_BLOCK);
        indices[o] = -1;
        continue;
      }
    }
    indices[o] = (int32_t)((int64_t)r * request_stride + (int64_t)block * block_size + e);
  }
}

}  // namespace
}  // namespace pa

extern "C" int64_t pa_selection_rows_per_request(int32_t topk, int32_t block_size, int32_t kv_len) {
  if (block_size < 1 || kv_len < 1 || topk < 0) return -1;
  const int64_t nb = ((int64_t)kv_len + block_size - 1) / block_size;
  if (topk > nb - 1) return -1;
  return (int64_t)topk * block_size + (kv_len - (nb - 1) * block_size);
}

extern "C" pa_status pa_sparse_csr(int32_t num_requests, int64_t per_request, int32_t* indptr,
                                   int32_t* last_page_len, int32_t* first_page_offset) {
  if (num_requests < 0 || per_request < 0 || !indptr || (num_requests > 0 && (!last_page_len || !first_page_offset)))
    return PA_EINVAL;
  if ((int64_t)num_requests * per_request > INT32_MAX) return PA_EINVAL;
  for (int32_t r = 0; r <= num_requests; ++r) indptr[r] = (int32_t)(r * per_request);
  for (int32_t r = 0; r < num_requests; ++r) {
    last_page_len[r] = per_request > 0 ? 1 : 0;
    first_page_offset[r] = 0;
  }
  return PA_OK;
}

extern "C" pa_status pa_selection_from_blocks(const int32_t* block_ids, int32_t num_requests, int32_t topk,
                                              int32_t block_size, int32_t kv_len, int64_t request_stride,
                                              int32_t* indices, int32_t* status, void* cuda_stream) {
  const int64_t per = pa_selection_rows_per_request(topk, block_size, kv_len);
  if (per < 0 || num_requests < 0 || request_stride < kv_len || !indices || (topk > 0 && !block_ids))
    return PA_EINVAL;
  if (num_requests == 0) return PA_OK;
  const int64_t total = (int64_t)num_requests * per;
  if (total > INT32_MAX || (int64_t)(num_requests - 1) * request_stride + kv_len - 1 > INT32_MAX)
    return PA_EUNSUPPORTED;
  const int32_t num_blocks = (int32_t)(((int64_t)kv_len + block_size - 1) / block_size);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PA_ECUDA;
  const int64_t want = (total + pa::kSelectThreads - 1) / pa::kSelectThreads;
  const int blocks = (int)(want < 8LL * sms ? want : 8LL * sms);
  const cudaError_t rc = pa::launch_dependent(pa::pa_selection_from_blocks_kernel, dim3(blocks),
                                              dim3(pa::kSelectThreads), 0, static_cast<cudaStream_t>(cuda_stream),
                                              block_ids, topk, block_size, num_blocks, (int32_t)per,
                                              (int32_t)total, request_stride, indices, status);
  return rc == cudaSuccess && cudaGetLastError() == cudaSuccess ? PA_OK : PA_ECUDA;
}
