// pa_plan.cpp -- host side of the C ABI: the decode plan, its reuse predicate,
// the q-heads-per-CTA helper and status strings.
//
// The plan follows PR #984 ("fused paged-attention decode v2 with CSR page
// table and cross-CTA split-KV"), What changed 4 (Plan), and issue #898
// ("Fused paged-attention decode v2: ..."), design piece 4: the chunk count
// sum_r max(1, ceil(pages_r / ppc)) is non-increasing in the chunk size ppc,
// so a binary search finds the largest ppc whose CTA count
// (chunks * Hkv * q_groups) still reaches the device target -- among the
// sizes that saturate the device, the one with the least merge work.  A
// floor keeps the chunk count within the 65535 grid bound; every request
// gets at least one chunk; chunks are emitted in request order.
#include <cstdint>
#include <cstring>
#include <vector>

#include "pa_v2.h"

namespace {

// Page sizes whose pages the kernel stages whole (<= 16 rows) or in 16-row slices.
bool page_size_ok(int32_t ps) { return (ps >= 1 && ps <= 16) || (ps > 16 && ps <= 256 && ps % 16 == 0); }

int64_t chunks_for(const std::vector<int64_t>& pages, int64_t ppc) {
  int64_t n = 0;
  for (int64_t p : pages) n += p > 0 ? (p + ppc - 1) / ppc : 1;
  return n;
}

uint64_t geometry_hash(const int32_t* indptr, int32_t batch) {
  // FNV-1a over the batch size and every request's page count.
  uint64_t h = 1469598103934665603ull;
  auto mix = [&h](int64_t v) {
    for (int i = 0; i < 8; ++i) {
      h ^= static_cast<uint64_t>((v >> (8 * i)) & 0xff);
      h *= 1099511628211ull;
    }
  };
  mix(batch);
  for (int32_t r = 0; r < batch; ++r) mix(static_cast<int64_t>(indptr[r + 1]) - indptr[r]);
  return h;
}

// Geometry rules of the CSR view (PR #984, What changed 1).  seq_lens may be null.
bool geometry_ok(const int32_t* indptr, const int32_t* lpl, const int32_t* fpo, const int32_t* seq_lens,
                 int32_t batch, int32_t ps) {
  if (indptr[0] != 0) return false;
  for (int32_t r = 0; r < batch; ++r) {
    int64_t pages = static_cast<int64_t>(indptr[r + 1]) - indptr[r];
    if (pages < 0) return false;
    if (pages == 0) {
      if (lpl[r] != 0 || fpo[r] != 0) return false;
    } else {
      if (lpl[r] < 1 || lpl[r] > ps) return false;
      if (fpo[r] < 0 || fpo[r] >= ps) return false;
      if (pages == 1 && fpo[r] >= lpl[r]) return false;
    }
    if (seq_lens) {
      int64_t L = pages == 0 ? 0 : (pages - 1) * ps + lpl[r] - fpo[r];
      if (L != seq_lens[r]) return false;
    }
  }
  return true;
}

}  // namespace

extern "C" {

pa_status pa_v2_plan(const int32_t* indptr, const int32_t* last_page_len, const int32_t* first_page_offset,
                     const int32_t* seq_lens, int32_t batch, int32_t page_size, int32_t num_qo_heads,
                     int32_t num_kv_heads, int32_t head_dim, int32_t kv_dtype, int32_t target_ctas,
                     int32_t pages_per_chunk_override, int32_t* request_indices, int32_t* kv_tile_indices,
                     int32_t cap_chunks, int32_t* o_indptr, pa_v2_plan_t* out) {
  if (!out || !indptr || !o_indptr || batch < 0 || cap_chunks < 0) return PA_EINVAL;
  if (batch > 0 && (!last_page_len || !first_page_offset)) return PA_EINVAL;
  if (cap_chunks > 0 && (!request_indices || !kv_tile_indices)) return PA_EINVAL;
  if (page_size < 1 || num_qo_heads < 1 || num_kv_heads < 1 || num_qo_heads % num_kv_heads != 0)
    return PA_EINVAL;
  if (pages_per_chunk_override < 0 || (pages_per_chunk_override == 0 && target_ctas < 1)) return PA_EINVAL;
  std::memset(out, 0, sizeof(*out));
  const int32_t group = num_qo_heads / num_kv_heads;
  const int32_t hpc = pa_v2_q_heads_per_cta(group, head_dim, kv_dtype);
  if (hpc == 0 || !page_size_ok(page_size)) return PA_EUNSUPPORTED;
  if (!geometry_ok(indptr, last_page_len, first_page_offset, seq_lens, batch, page_size)) return PA_EGEOMETRY;
  const int32_t q_groups = (group + hpc - 1) / hpc;
  if (static_cast<int64_t>(num_kv_heads) * q_groups > 65535) return PA_EUNSUPPORTED;

  std::vector<int64_t> pages(batch);
  int64_t hi = 1;
  for (int32_t r = 0; r < batch; ++r) {
    pages[r] = static_cast<int64_t>(indptr[r + 1]) - indptr[r];
    if (pages[r] > hi) hi = pages[r];
  }
  if (chunks_for(pages, hi) > PA_V2_MAX_CHUNKS) return PA_EINVAL;  // more requests than launchable chunks
  // lo: smallest chunk size whose chunk count fits the grid bound.
  int64_t a = 1, b = hi;
  while (a < b) {
    int64_t mid = a + (b - a) / 2;
    if (chunks_for(pages, mid) <= PA_V2_MAX_CHUNKS) b = mid; else a = mid + 1;
  }
  const int64_t lo = a;
  const int64_t per_chunk = static_cast<int64_t>(num_kv_heads) * q_groups;
  int64_t ppc;
  if (pages_per_chunk_override > 0) {
    if (chunks_for(pages, pages_per_chunk_override) > PA_V2_MAX_CHUNKS) return PA_EINVAL;
    ppc = pages_per_chunk_override;
  } else if (chunks_for(pages, lo) * per_chunk < target_ctas) {
    ppc = lo;  // the target is out of reach: take the most parallel launchable plan
  } else {
    // largest ppc in [lo, hi] with chunks(ppc) * per_chunk >= target
    a = lo;
    b = hi;
    while (a < b) {
      int64_t mid = a + (b - a + 1) / 2;
      if (chunks_for(pages, mid) * per_chunk >= target_ctas) a = mid; else b = mid - 1;
    }
    ppc = a;
  }
  const int64_t n = chunks_for(pages, ppc);

  int64_t nnz = batch > 0 ? indptr[batch] : 0;
  out->batch = batch;
  out->num_qo_heads = num_qo_heads;
  out->num_kv_heads = num_kv_heads;
  out->head_dim = head_dim;
  out->page_size = page_size;
  out->kv_dtype = kv_dtype;
  out->q_heads_per_cta = hpc;
  out->q_groups = q_groups;
  out->pages_per_chunk = static_cast<int32_t>(ppc);
  out->lo_pages_per_chunk = static_cast<int32_t>(lo);
  out->hi_pages_per_chunk = static_cast<int32_t>(hi);
  out->num_chunks = static_cast<int32_t>(n);
  out->needs_merge = n > batch ? 1 : 0;
  out->target_ctas = target_ctas;
  out->total_ctas = static_cast<int32_t>(n * per_chunk);
  out->num_indices = nnz;
  out->workspace_v_bytes = n * num_qo_heads * static_cast<int64_t>(head_dim) * 4;
  out->workspace_lse_bytes = n * num_qo_heads * 4;
  out->counter_bytes = static_cast<int64_t>(batch) * per_chunk * 4;
  out->stack_members = 1;
  out->out_row_step = 1;
  out->geometry_hash = geometry_hash(indptr, batch);
  if (n > cap_chunks) return PA_ECAPACITY;

  int64_t c = 0;
  o_indptr[0] = 0;
  for (int32_t r = 0; r < batch; ++r) {
    int64_t nr = pages[r] > 0 ? (pages[r] + ppc - 1) / ppc : 1;
    for (int64_t t = 0; t < nr; ++t, ++c) {
      request_indices[c] = r;
      kv_tile_indices[c] = static_cast<int32_t>(t);
    }
    o_indptr[r + 1] = static_cast<int32_t>(c);
  }
  return PA_OK;
}

int32_t pa_v2_plan_matches(const pa_v2_plan_t* plan, const int32_t* indptr, const int32_t* last_page_len,
                           const int32_t* first_page_offset, int32_t batch) {
  if (!plan || !indptr || batch != plan->batch) return 0;
  if (batch > 0 && (!last_page_len || !first_page_offset)) return 0;
  if (!geometry_ok(indptr, last_page_len, first_page_offset, nullptr, batch, plan->page_size)) return 0;
  if (batch > 0 && indptr[batch] != plan->num_indices) return 0;
  return geometry_hash(indptr, batch) == plan->geometry_hash ? 1 : 0;
}

pa_status pa_status_from_device(int32_t w) {
  if (w == 0) return PA_OK;
  if (w & PA_DEVICE_WAIT_TIMEOUT) return PA_ECUDA;
  return PA_EOOB;
}

const char* pa_status_string(int32_t s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_EINVAL: return "PA_EINVAL: invalid argument (null pointer, bad size or misaligned buffer)";
    case PA_EGEOMETRY: return "PA_EGEOMETRY: CSR page table breaks the geometry rules";
    case PA_ECAPACITY: return "PA_ECAPACITY: chunk arrays too small (plan.num_chunks holds the need)";
    case PA_EUNSUPPORTED: return "PA_EUNSUPPORTED: head_dim / dtype / page_size not served";
    case PA_ECUDA: return "PA_ECUDA: CUDA call or launch failed";
    case PA_EOOB: return "PA_EOOB: device-side index out of range";
    default: return "unknown pa_status";
  }
}

// The smallest chunk size whose CTAs fit one wave.  The plan's binary search
// takes the largest chunk size that still reaches the target, so its CTA count
// may pass the target by up to one chunk per request; with one CTA per SM the
// extra CTAs then run as a second, almost empty wave.  CTA count of a size s:
// sum over requests of max(1, ceil(pages_r / s)) * ctas_per_chunk.
int32_t pa_v2_wave_fit_pages_per_chunk(const int32_t* indptr, int32_t batch, int32_t ctas_per_chunk,
                                       int32_t wave) {
  if (!indptr || batch < 1 || ctas_per_chunk < 1 || wave < 1 || indptr[0] != 0) return 0;
  int32_t longest = 1;
  for (int32_t r = 0; r < batch; ++r) {
    const int32_t n = indptr[r + 1] - indptr[r];
    if (n < 0) return 0;
    if (n > longest) longest = n;
  }
  auto ctas = [&](int32_t size) {
    int64_t chunks = 0;
    for (int32_t r = 0; r < batch; ++r) {
      const int64_t n = indptr[r + 1] - indptr[r];
      chunks += n <= size ? 1 : (n + size - 1) / size;
    }
    return chunks * ctas_per_chunk;
  };
  if (ctas(longest) > wave) return longest;  // one chunk per request does not fit either
  int32_t lo = 1, hi = longest;
  while (lo < hi) {
    const int32_t mid = lo + (hi - lo) / 2;
    if (ctas(mid) <= wave)
      hi = mid;
    else
      lo = mid + 1;
  }
  return lo;
}

// A chunk size that gives every warp of the tensor-core partial kernel the same
// number of stages.  That kernel stages 16 pool rows at a time -- floor(16 /
// page_size) whole pages when page_size <= 16, a 16-row slice of a page when
// page_size is a multiple of 16 -- and its 8 warps take a chunk's stages in
// turn, so a launch ends with the busiest warp: at 32768 tokens of 16-row pages
// the plan's 113 pages per chunk leave one warp a 15th stage, 112 = 8 x 14 do
// not.  Scans down from `pages_per_chunk` for the largest size whose stage
// count is a multiple of 8 and whose chunk count (sum over requests of
// max(1, ceil(pages_r / size))) is still that of `pages_per_chunk`.
constexpr int32_t kBalanceStageRows = 16;  // rows per stage (pa_internal.cuh kStageRows)
constexpr int32_t kBalanceWarps = 8;       // warps per CTA of the tensor-core kernel

int32_t pa_v2_balanced_pages_per_chunk(const int32_t* indptr, int32_t batch, int32_t page_size,
                                       int32_t pages_per_chunk) {
  if (!indptr || batch < 1 || page_size < 1 || pages_per_chunk < 1 || indptr[0] != 0) return 0;
  for (int32_t r = 0; r < batch; ++r)
    if (indptr[r + 1] < indptr[r]) return 0;
  if (page_size > kBalanceStageRows && page_size % kBalanceStageRows != 0) return pages_per_chunk;
  auto stages = [&](int64_t size) -> int64_t {
    if (page_size <= kBalanceStageRows) {
      const int64_t per = kBalanceStageRows / page_size;
      return (size + per - 1) / per;
    }
    return size * (page_size / kBalanceStageRows);
  };
  auto chunks = [&](int64_t size) {
    int64_t n = 0;
    for (int32_t r = 0; r < batch; ++r) {
      const int64_t pages = indptr[r + 1] - indptr[r];
      n += pages <= size ? 1 : (pages + size - 1) / size;
    }
    return n;
  };
  const int64_t want = chunks(pages_per_chunk);
  // the chunk count does not decrease as the size shrinks: stop at the first size that adds a chunk
  for (int64_t size = pages_per_chunk; size >= 1; --size) {
    if (stages(size) % kBalanceWarps != 0) continue;
    if (chunks(size) != want) break;
    return static_cast<int32_t>(size);
  }
  return pages_per_chunk;
}

const char* pa_version(void) { return "pa_v2 0.1 (sm_103a)"; }

}  // extern "C"
