// pa_launch.h -- internal launch entry points shared between translation units
// of the library (host code only; not part of the C ABI).
#pragma once

#include <cstdint>

#include "pa_v2.h"

namespace pa {

// pa_v2_decode_partial for a launch that nothing runs before on the GPU (the
// first kernel of a host step): the same kernel without its pre-wait L2
// warm-up, whose speculative reads could only add latency there (more so when
// the page table is host memory read over NVLink-C2C).
pa_status decode_partial_leading(const pa_v2_plan_t* plan, const float* q, const void* k_pool, const void* v_pool,
                                 int32_t kv_dtype, int64_t num_pages, const int32_t* indices, int64_t num_indices,
                                 const int32_t* indptr, const int32_t* last_page_len,
                                 const int32_t* first_page_offset, const int32_t* request_indices,
                                 const int32_t* kv_tile_indices, float sm_scale, float* v_out, float* lse2_out,
                                 int32_t* status, void* cuda_stream);

}  // namespace pa
