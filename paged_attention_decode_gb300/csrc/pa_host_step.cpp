// pa_host_step.cpp -- one whole decode step for callers whose per-step inputs
// live in host memory: check the cached plan, copy the inputs in, run the
// partial kernel (and the merge when the plan needs one), copy the outputs
// back and wait, in one call.
//
// The pages time the decode with the plan built once outside the step and the
// query cast once outside the timed region (PR #984, the commit extending
// examples/page_gather_microbench.rs); what changes every step is the query
// and the page table.  A caller that keeps those on the host otherwise pays
// several API calls per step; here the inputs travel as one packed buffer in
// one host-to-device copy and the outputs (with the device status word) in one
// device-to-host copy, on the caller's stream.
//
// The mapped variants drop both copies.  On a GB300 the Grace CPU's memory is
// reachable from the GPU over the coherent NVLink-C2C link, so the kernels read
// the packed inputs straight out of the caller's page-locked host_in and the
// last kernel writes the status, out and lse2 straight into host_out: each step
// is then two kernel launches, the second a programmatic dependent of the first,
// instead of copy -> partial -> merge -> copy with a full dependency at either
// copy.  The merge also counts its finished CTAs into the status slot, and the
// host waits for that count instead of synchronising the stream: the results
// are in host memory before the launch has formally completed.
#include <cuda_runtime.h>

#include <atomic>
#include <chrono>
#include <cstdint>
#include <cstring>

#include "pa_launch.h"
#include "pa_v2.h"

namespace {

int64_t round16(int64_t x) { return (x + 15) & ~int64_t{15}; }

}  // namespace

extern "C" pa_status pa_v2_host_io_layout(const pa_v2_plan_t* plan, int64_t* in_bytes, int64_t* out_bytes,
                                          int64_t* io_bytes) {
  if (!plan || !in_bytes || !out_bytes || !io_bytes || plan->batch < 0) return PA_EINVAL;
  const int64_t B = plan->batch;
  const int64_t rows = B * plan->num_qo_heads;
  const int64_t words = rows * plan->head_dim + plan->num_indices + (B + 1) + 2 * B;
  *in_bytes = round16(words * 4) + 16;                     // inputs, then a zeroed 16-byte status slot
  *out_bytes = 16 + rows * plan->head_dim * 4 + rows * 4;  // the status slot, out, lse2
  *io_bytes = *in_bytes - 16 + *out_bytes;                 // the status slot is shared
  return PA_OK;
}

namespace {

// The device address of a page-locked, mapped host buffer (16-byte aligned), or
// null.
unsigned char* mapped_address(const void* host) {
  if (!host || (reinterpret_cast<uintptr_t>(host) & 15u)) return nullptr;
  void* dev = nullptr;
  if (cudaHostGetDevicePointer(&dev, const_cast<void*>(host), 0) != cudaSuccess || !dev) {
    cudaGetLastError();
    return nullptr;
  }
  return static_cast<unsigned char*>(dev);
}

// Queue one host step on `stream` without waiting: the input copy, the partial
// kernel (and the merge when the plan needs one), the output copy.  Checks the
// arguments and the plan against the step's page table first.  With `mapped`
// (the device addresses of host_in and host_out, from mapped_address): no
// copies; the kernels read and write those, the status word is host_out's,
// which the caller zeroes before the step, dev_io is not used, and the merge
// counts its finished CTAs into the slot's second word (*merge_ctas of them; 0
// when the step has no merge and the caller must synchronise instead).
pa_status enqueue_host_step(const pa_v2_plan_t* plan, const void* host_in, void* host_out, void* dev_io,
                            const void* k_pool, const void* v_pool, int32_t kv_dtype, int64_t num_pages,
                            const int32_t* request_indices, const int32_t* kv_tile_indices, const int32_t* o_indptr,
                            float sm_scale, float* workspace_v, float* workspace_lse, cudaStream_t stream,
                            bool check_geometry, unsigned char* const* mapped, int64_t* merge_ctas) {
  *merge_ctas = 0;
  int64_t in_bytes = 0, out_bytes = 0, io_bytes = 0;
  if (pa_v2_host_io_layout(plan, &in_bytes, &out_bytes, &io_bytes) != PA_OK) return PA_EINVAL;
  if (!host_in || !host_out) return PA_EINVAL;
  if (!mapped && (!dev_io || (reinterpret_cast<uintptr_t>(dev_io) & 15u))) return PA_EINVAL;
  if (plan->needs_merge && (!workspace_v || !workspace_lse || !o_indptr)) return PA_EINVAL;
  const int32_t B = plan->batch;
  const int64_t rows = (int64_t)B * plan->num_qo_heads;
  const int64_t q_words = rows * plan->head_dim;

  // the packed host inputs: q | indices | indptr | last_page_len | first_page_offset (4-byte words)
  const int32_t* h_words = static_cast<const int32_t*>(host_in);
  const int32_t* h_indptr = h_words + q_words + plan->num_indices;
  const int32_t* h_lpl = h_indptr + B + 1;
  const int32_t* h_fpo = h_lpl + B;
  if (check_geometry && !pa_v2_plan_matches(plan, h_indptr, h_lpl, h_fpo, B)) return PA_EGEOMETRY;

  const unsigned char* in_region;  // the packed inputs as the kernels address them
  unsigned char* out_region;       // the status slot, then out, lse2
  if (mapped) {
    in_region = mapped[0];
    out_region = mapped[1];
    if (!in_region || !out_region) return PA_EINVAL;
  } else {
    unsigned char* io = static_cast<unsigned char*>(dev_io);
    in_region = io;
    if (cudaMemcpyAsync(io, host_in, (size_t)in_bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
      return PA_ECUDA;
    out_region = io + in_bytes - 16;  // the status slot the copy above zeroed
  }

  const float* q = reinterpret_cast<const float*>(in_region);
  const int32_t* indices = reinterpret_cast<const int32_t*>(in_region) + q_words;
  const int32_t* indptr = indices + plan->num_indices;
  const int32_t* lpl = indptr + B + 1;
  const int32_t* fpo = lpl + B;
  int32_t* status = reinterpret_cast<int32_t*>(out_region);
  float* out = reinterpret_cast<float*>(out_region + 16);
  float* lse = out + q_words;
  void* cs = static_cast<void*>(stream);

  pa_status rc;
  if (plan->needs_merge) {
    rc = pa::decode_partial_leading(plan, q, k_pool, v_pool, kv_dtype, num_pages, indices, plan->num_indices, indptr,
                                    lpl, fpo, request_indices, kv_tile_indices, sm_scale, workspace_v, workspace_lse,
                                    status, cs);
    if (rc == PA_OK)
      rc = pa::launch_merge(workspace_v, workspace_lse, o_indptr, B, plan->num_chunks, plan->num_qo_heads,
                            plan->head_dim, out, lse, status, mapped ? status + 1 : nullptr,
                            mapped ? merge_ctas : nullptr, cs);
  } else {
    rc = pa::decode_partial_leading(plan, q, k_pool, v_pool, kv_dtype, num_pages, indices, plan->num_indices, indptr,
                                    lpl, fpo, request_indices, kv_tile_indices, sm_scale, out, lse, status, cs);
  }
  if (rc != PA_OK) return rc;
  if (!mapped &&
      cudaMemcpyAsync(host_out, out_region, (size_t)out_bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return PA_ECUDA;
  return PA_OK;
}

void clear_status_slot(void* host_out) { std::memset(host_out, 0, 16); }

// Wait for the merge's count of finished CTAs in host_out's status slot to reach
// `ctas` (each CTA adds one after a system-scope fence behind its stores), then
// order the reads that follow after it.  False after ~5 s without it.
bool wait_merge_count(const void* host_out, int64_t ctas) {
  const volatile int32_t* count =
      reinterpret_cast<const volatile int32_t*>(static_cast<const unsigned char*>(host_out) + 4);
  const auto t0 = std::chrono::steady_clock::now();
  for (uint32_t i = 1;; ++i) {
    if (*count >= ctas) {
      std::atomic_thread_fence(std::memory_order_acquire);
      return true;
    }
    if ((i & 4095u) == 0 && std::chrono::steady_clock::now() - t0 > std::chrono::seconds(5)) return false;
  }
}

// The end of a host step: wait for the merge's count when there is one (the
// stream is then left to retire the step's kernels on its own), else, or when
// the count never comes, synchronise the stream; then the status word.
pa_status finish_host_step(cudaStream_t stream, const void* host_out, int64_t merge_ctas) {
  if (merge_ctas <= 0 || !wait_merge_count(host_out, merge_ctas)) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return PA_ECUDA;
  }
  int32_t word = 0;
  std::memcpy(&word, host_out, sizeof(word));
  return pa_status_from_device(word);
}

pa_status decode_host(const pa_v2_plan_t* plan, const void* host_in, void* host_out, void* dev_io,
                      const void* k_pool, const void* v_pool, int32_t kv_dtype, int64_t num_pages,
                      const int32_t* request_indices, const int32_t* kv_tile_indices, const int32_t* o_indptr,
                      float sm_scale, float* workspace_v, float* workspace_lse, void* cuda_stream, bool mapped) {
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  unsigned char* addr[2] = {nullptr, nullptr};
  if (mapped) {
    addr[0] = mapped_address(host_in);
    addr[1] = mapped_address(host_out);
    if (addr[1]) clear_status_slot(host_out);
  }
  int64_t merge_ctas = 0;
  const pa_status rc = enqueue_host_step(plan, host_in, host_out, dev_io, k_pool, v_pool, kv_dtype, num_pages,
                                         request_indices, kv_tile_indices, o_indptr, sm_scale, workspace_v,
                                         workspace_lse, stream, true, mapped ? addr : nullptr, &merge_ctas);
  if (rc != PA_OK) {
    cudaStreamSynchronize(stream);  // a copy or kernel already queued may still be reading host_in
    return rc;
  }
  return finish_host_step(stream, host_out, merge_ctas);
}

}  // namespace

extern "C" pa_status pa_v2_decode_host(const pa_v2_plan_t* plan, const void* host_in, void* host_out, void* dev_io,
                                       const void* k_pool, const void* v_pool, int32_t kv_dtype, int64_t num_pages,
                                       const int32_t* request_indices, const int32_t* kv_tile_indices,
                                       const int32_t* o_indptr, float sm_scale, float* workspace_v,
                                       float* workspace_lse, void* cuda_stream) {
  return decode_host(plan, host_in, host_out, dev_io, k_pool, v_pool, kv_dtype, num_pages, request_indices,
                     kv_tile_indices, o_indptr, sm_scale, workspace_v, workspace_lse, cuda_stream, false);
}

extern "C" pa_status pa_v2_decode_host_mapped(const pa_v2_plan_t* plan, const void* host_in, void* host_out,
                                              const void* k_pool, const void* v_pool, int32_t kv_dtype,
                                              int64_t num_pages, const int32_t* request_indices,
                                              const int32_t* kv_tile_indices, const int32_t* o_indptr,
                                              float sm_scale, float* workspace_v, float* workspace_lse,
                                              void* cuda_stream) {
  return decode_host(plan, host_in, host_out, nullptr, k_pool, v_pool, kv_dtype, num_pages, request_indices,
                     kv_tile_indices, o_indptr, sm_scale, workspace_v, workspace_lse, cuda_stream, true);
}

// ---- the same step as one CUDA graph ---------------------------------------
//
// Per step the direct call above issues two copies and two launches through
// the runtime; the graph replays them with one launch.  Everything except the
// contents of host_in is bound when the graph is made: the plan (a copy), the
// buffers, the pools, the chunk arrays, the scale.  Capture runs on a private
// stream; the programmatic launches of the partial and merge kernels become
// programmatic edges of the graph.

struct pa_v2_host_graph {
  pa_v2_plan_t plan;
  const void* host_in;
  void* host_out;
  bool mapped;         // the status slot is host_out's, zeroed by run()
  int64_t merge_ctas;  // mapped: the merge CTAs run() waits to see counted (0: synchronise)
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};

namespace {

pa_status host_graph_create(const pa_v2_plan_t* plan, const void* host_in, void* host_out, void* dev_io,
                            const void* k_pool, const void* v_pool, int32_t kv_dtype, int64_t num_pages,
                            const int32_t* request_indices, const int32_t* kv_tile_indices, const int32_t* o_indptr,
                            float sm_scale, float* workspace_v, float* workspace_lse, bool mapped,
                            pa_v2_host_graph_t** out) {
  if (!plan || !out) return PA_EINVAL;
  *out = nullptr;
  // resolved before the capture, which admits only stream work
  unsigned char* addr[2] = {nullptr, nullptr};
  if (mapped) {
    addr[0] = mapped_address(host_in);
    addr[1] = mapped_address(host_out);
    if (!addr[0] || !addr[1]) return PA_EINVAL;
  }
  cudaStream_t cap = nullptr;
  if (cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking) != cudaSuccess) return PA_ECUDA;
  if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaStreamDestroy(cap);
    return PA_ECUDA;
  }
  // the geometry is checked on every run, against that step's page table
  int64_t merge_ctas = 0;
  pa_status rc = enqueue_host_step(plan, host_in, host_out, dev_io, k_pool, v_pool, kv_dtype, num_pages,
                                   request_indices, kv_tile_indices, o_indptr, sm_scale, workspace_v, workspace_lse,
                                   cap, false, mapped ? addr : nullptr, &merge_ctas);
  cudaGraph_t graph = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(cap, &graph);
  cudaStreamDestroy(cap);
  if (rc == PA_OK && (ec != cudaSuccess || !graph)) rc = PA_ECUDA;
  cudaGraphExec_t exec = nullptr;
  if (rc == PA_OK && cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) rc = PA_ECUDA;
  if (rc != PA_OK) {
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();
    return rc;
  }
  pa_v2_host_graph_t* g = new pa_v2_host_graph_t;
  g->plan = *plan;
  g->host_in = host_in;
  g->host_out = host_out;
  g->mapped = mapped;
  g->merge_ctas = merge_ctas;
  g->graph = graph;
  g->exec = exec;
  *out = g;
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_v2_host_graph_create(const pa_v2_plan_t* plan, const void* host_in, void* host_out,
                                             void* dev_io, const void* k_pool, const void* v_pool, int32_t kv_dtype,
                                             int64_t num_pages, const int32_t* request_indices,
                                             const int32_t* kv_tile_indices, const int32_t* o_indptr, float sm_scale,
                                             float* workspace_v, float* workspace_lse, pa_v2_host_graph_t** out) {
  return host_graph_create(plan, host_in, host_out, dev_io, k_pool, v_pool, kv_dtype, num_pages, request_indices,
                           kv_tile_indices, o_indptr, sm_scale, workspace_v, workspace_lse, false, out);
}

extern "C" pa_status pa_v2_host_graph_create_mapped(const pa_v2_plan_t* plan, const void* host_in, void* host_out,
                                                    const void* k_pool, const void* v_pool, int32_t kv_dtype,
                                                    int64_t num_pages, const int32_t* request_indices,
                                                    const int32_t* kv_tile_indices, const int32_t* o_indptr,
                                                    float sm_scale, float* workspace_v, float* workspace_lse,
                                                    pa_v2_host_graph_t** out) {
  return host_graph_create(plan, host_in, host_out, nullptr, k_pool, v_pool, kv_dtype, num_pages, request_indices,
                           kv_tile_indices, o_indptr, sm_scale, workspace_v, workspace_lse, true, out);
}

extern "C" pa_status pa_v2_host_graph_run(pa_v2_host_graph_t* g, void* cuda_stream) {
  if (!g) return PA_EINVAL;
  const pa_v2_plan_t* plan = &g->plan;
  const int32_t B = plan->batch;
  const int32_t* h_words = static_cast<const int32_t*>(g->host_in);
  const int32_t* h_indptr = h_words + (int64_t)B * plan->num_qo_heads * plan->head_dim + plan->num_indices;
  if (!pa_v2_plan_matches(plan, h_indptr, h_indptr + B + 1, h_indptr + 2 * B + 1, B)) return PA_EGEOMETRY;
  if (g->mapped) clear_status_slot(g->host_out);
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  if (cudaGraphLaunch(g->exec, stream) != cudaSuccess) {
    cudaStreamSynchronize(stream);
    return PA_ECUDA;
  }
  return finish_host_step(stream, g->host_out, g->mapped ? g->merge_ctas : 0);
}

extern "C" void pa_v2_host_graph_destroy(pa_v2_host_graph_t* g) {
  if (!g) return;
  cudaGraphExecDestroy(g->exec);
  cudaGraphDestroy(g->graph);
  delete g;
}
