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

// pa_merge_states with an optional completion count: `done` (or null) is an
// int32 in memory the host can read -- a word of a mapped host buffer -- to which
// every CTA adds one after a system-scope fence that follows its stores, so the
// count reaching *ctas (the CTAs launched; 0 when nothing was) means every result
// of the merge, and every status bit of the kernels before it, is visible to the
// host.  Same checks and errors as pa_merge_states.
pa_status launch_merge(const float* v_in, const float* lse2_in, const int32_t* o_indptr, int32_t num_rows_out,
                       int32_t num_partials, int32_t num_heads, int32_t head_dim, float* v_out, float* lse2_out,
                       int32_t* status, int32_t* done, int64_t* ctas, void* cuda_stream);

}  // namespace pa
