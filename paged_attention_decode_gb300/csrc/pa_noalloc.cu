// pa_noalloc.cu -- pa_v2_decode for callers that cannot allocate device memory.
//
// Some users of this library run inside a process that owns every device
// allocation: a serving engine that reserves the GPU's memory up front for its
// own pools, or a plugin that its host hands only input and output pointers.
// They cannot call cudaMalloc for the partial workspace and the ticket
// counters that pa_v2_decode takes from its caller.  This entry point takes
// them from a fixed array compiled into the library instead and allocates
// nothing.  (The pages have no counterpart to it.)
//
// The array: PA_V2_NOALLOC_SCRATCH_BYTES (8 MiB) of device memory per GPU that
// loads the library, held until the process exits.  Host code cannot use the
// array's name as a device address (on the host it names a stand-in), so the
// first call on each device asks the runtime for that device's address with
// the device current, and remembers it for the life of the process (so the
// address is stale after a cudaDeviceReset of that device).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "pa_v2.h"

namespace {

constexpr size_t kScratchBytes = PA_V2_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

size_t round256(int64_t x) { return (static_cast<size_t>(x) + 255u) & ~static_cast<size_t>(255u); }

// Device address of g_noalloc_scratch on `device` (which must be current), or
// nullptr if the runtime cannot provide it.
void* scratch_on(int device) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  if (device < 0 || device >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[device]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();  // leave no sticky-looking error behind for the caller's next check
      return nullptr;
    }
    addr[device] = p;
  }
  return addr[device];
}

}  // namespace

extern "C" pa_status pa_v2_decode_noalloc(const pa_v2_plan_t* plan, const float* q, const void* k_pool,
                                          const void* v_pool, int32_t kv_dtype, int64_t num_pages,
                                          const int32_t* indices, int64_t num_indices, const int32_t* indptr,
                                          const int32_t* last_page_len, const int32_t* first_page_offset,
                                          const int32_t* request_indices, const int32_t* kv_tile_indices,
                                          const int32_t* o_indptr, float sm_scale, float* out, float* lse2_out,
                                          int32_t* status, void* cuda_stream) {
  if (!plan || plan->counter_bytes < 0 || plan->workspace_v_bytes < 0 || plan->workspace_lse_bytes < 0)
    return PA_EINVAL;
  const size_t counters_at = 0;
  const size_t v_at = counters_at + round256(plan->counter_bytes);
  const size_t lse_at = v_at + round256(plan->workspace_v_bytes);
  const size_t end = lse_at + round256(plan->workspace_lse_bytes);
  if (end > kScratchBytes) return PA_ECAPACITY;
  if (plan->num_chunks == 0) return PA_OK;

  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PA_ECUDA;
  unsigned char* base = static_cast<unsigned char*>(scratch_on(device));
  if (!base) return PA_ECUDA;
  int32_t* counters = reinterpret_cast<int32_t*>(base + counters_at);
  float* workspace_v = reinterpret_cast<float*>(base + v_at);
  float* workspace_lse = reinterpret_cast<float*>(base + lse_at);

  // The counters must start at zero; the array keeps whatever the previous call left.
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  if (plan->counter_bytes > 0 &&
      cudaMemsetAsync(counters, 0, static_cast<size_t>(plan->counter_bytes), stream) != cudaSuccess)
    return PA_ECUDA;
  return pa_v2_decode(plan, q, k_pool, v_pool, kv_dtype, num_pages, indices, num_indices, indptr, last_page_len,
                      first_page_offset, request_indices, kv_tile_indices, o_indptr, sm_scale, workspace_v,
                      workspace_lse, counters, out, lse2_out, nullptr, nullptr, status, cuda_stream);
}
