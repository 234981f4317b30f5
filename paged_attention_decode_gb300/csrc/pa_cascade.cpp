// pa_cascade.cpp -- host side of cascade decode: shared-prefix detection and
// the split of a batch into the two cascade levels.
//
// cascade-attention.md (issue #903).  Detection reads the CSR page table, not
// pool refcounts: two requests whose page i is the same physical page share
// those bytes.  Requests whose window starts mid-page are left out (the span
// would not be whole pages).  The rest are grouped by their first page; a
// group's shared span is the run of leading positions on which all its members
// hold the same page, capped at pages - 1 for every member (only a last page
// may be partly filled, and level 0 declares its pages full); the group that
// removes the most page reads, shared * (members - 1), wins, subject to the
// minimum span and member count.  Requests outside the winning group keep their
// whole range at level 1 and merge as a single row (the identity).
#include <algorithm>
#include <cstdint>
#include <unordered_map>
#include <vector>

#include "pa_v2.h"

extern "C" pa_status pa_v2_cascade_detect(const int32_t* indptr, const int32_t* indices,
                                          const int32_t* first_page_offset, int32_t batch, int32_t min_shared_pages,
                                          int32_t min_members, int32_t* member_of, int32_t* num_members,
                                          int32_t* shared_pages) {
  if (!indptr || batch < 0 || !num_members || !shared_pages || (batch > 0 && (!first_page_offset || !member_of)))
    return PA_EINVAL;
  *num_members = 0;
  *shared_pages = 0;
  for (int32_t r = 0; r < batch; ++r) member_of[r] = 0;
  if (batch > 0 && indptr[batch] > 0 && !indices) return PA_EINVAL;
  if (indptr[0] != 0) return PA_EGEOMETRY;
  for (int32_t r = 0; r < batch; ++r)
    if (indptr[r + 1] < indptr[r]) return PA_EGEOMETRY;

  // group eligible requests by first page, remembering the order groups appear in
  std::unordered_map<int32_t, int32_t> group_of;
  std::vector<std::vector<int32_t>> groups;
  for (int32_t r = 0; r < batch; ++r) {
    const int32_t pages = indptr[r + 1] - indptr[r];
    if (first_page_offset[r] != 0 || pages < 2) continue;
    const int32_t key = indices[indptr[r]];
    auto it = group_of.find(key);
    if (it == group_of.end()) {
      group_of.emplace(key, static_cast<int32_t>(groups.size()));
      groups.push_back({r});
    } else {
      groups[it->second].push_back(r);
    }
  }
  int64_t best_score = -1;
  int32_t best = -1, best_shared = 0;
  for (int32_t g = 0; g < static_cast<int32_t>(groups.size()); ++g) {
    const auto& mem = groups[g];
    if (mem.size() < 2) continue;
    int32_t cap = INT32_MAX;
    for (int32_t r : mem) cap = std::min(cap, indptr[r + 1] - indptr[r] - 1);
    const int32_t* first = indices + indptr[mem[0]];
    int32_t shared = 0;
    for (; shared < cap; ++shared) {
      bool same = true;
      for (int32_t r : mem)
        if (indices[indptr[r] + shared] != first[shared]) {
          same = false;
          break;
        }
      if (!same) break;
    }
    const int64_t score = static_cast<int64_t>(shared) * (static_cast<int64_t>(mem.size()) - 1);
    if (score > best_score) {
      best_score = score;
      best = g;
      best_shared = shared;
    }
  }
  const int32_t need = min_members > 2 ? min_members : 2;
  if (best < 0 || static_cast<int32_t>(groups[best].size()) < need || best_shared < min_shared_pages) return PA_OK;
  for (int32_t r : groups[best]) member_of[r] = 1;
  *num_members = static_cast<int32_t>(groups[best].size());
  *shared_pages = best_shared;
  return PA_OK;
}

extern "C" pa_status pa_v2_cascade_split(const int32_t* indptr, const int32_t* indices, const int32_t* last_page_len,
                                         const int32_t* first_page_offset, int32_t batch, const int32_t* member_of,
                                         int32_t shared_pages, int32_t* l1_indptr, int32_t* l1_indices,
                                         int32_t* l1_last_page_len, int32_t* l1_first_page_offset,
                                         int32_t* member_rows, int32_t* l0_out_rows, int32_t* l1_out_rows,
                                         int32_t* merge_indptr) {
  if (!indptr || batch < 0 || shared_pages < 0 || !l1_indptr || !merge_indptr) return PA_EINVAL;
  if (batch > 0 && (!last_page_len || !first_page_offset || !member_of || !l1_last_page_len ||
                    !l1_first_page_offset || !l1_out_rows))
    return PA_EINVAL;
  int32_t members = 0;
  for (int32_t r = 0; r < batch; ++r) {
    if (!member_of[r]) continue;
    const int32_t pages = indptr[r + 1] - indptr[r];
    if (first_page_offset[r] != 0 || shared_pages > pages - 1) return PA_EGEOMETRY;
    ++members;
  }
  if (members > 0 && (!member_rows || !l0_out_rows)) return PA_EINVAL;
  l1_indptr[0] = 0;
  merge_indptr[0] = 0;
  int32_t m = 0;
  for (int32_t r = 0; r < batch; ++r) {
    const int32_t skip = member_of[r] ? shared_pages : 0;
    const int32_t n = indptr[r + 1] - indptr[r] - skip;
    for (int32_t i = 0; i < n; ++i) l1_indices[l1_indptr[r] + i] = indices[indptr[r] + skip + i];
    l1_indptr[r + 1] = l1_indptr[r] + n;
    l1_last_page_len[r] = last_page_len[r];
    l1_first_page_offset[r] = first_page_offset[r];
    merge_indptr[r + 1] = merge_indptr[r] + (member_of[r] ? 2 : 1);
    if (member_of[r]) {
      member_rows[m] = r;
      l0_out_rows[m] = merge_indptr[r];  // level 0 takes the first row of the member's group
      ++m;
    }
    l1_out_rows[r] = merge_indptr[r + 1] - 1;  // level 1 takes the last row of every group
  }
  return PA_OK;
}


// The two cascade levels planned for one launch (cascade-attention.md): one chunk size for both levels,
// the smallest whose CTAs fit the wave, so that no CTA of the launch reads more pages than another; and the
// merge input laid out request by request (level-0 chunks of a member, then its level-1 chunks), so that one
// merge folds every request's states.
extern "C" pa_status pa_v2_cascade_plan(int32_t members, int32_t shared_pages, const int32_t* l1_indptr,
                                        const int32_t* l1_last_page_len, const int32_t* l1_first_page_offset,
                                        const int32_t* l1_seq_lens, int32_t l1_batch, const int32_t* member_requests,
                                        int32_t page_size, int32_t num_qo_heads, int32_t num_kv_heads,
                                        int32_t head_dim, int32_t kv_dtype, int32_t wave_ctas,
                                        int32_t* l0_request_indices, int32_t* l0_kv_tile_indices,
                                        int32_t l0_cap_chunks, int32_t* l0_o_indptr, int32_t* l1_request_indices,
                                        int32_t* l1_kv_tile_indices, int32_t l1_cap_chunks, int32_t* l1_o_indptr,
                                        int32_t* l0_part_rows, int32_t* l1_part_rows, int32_t* merge_indptr,
                                        pa_v2_plan_t* plan0, pa_v2_plan_t* plan1) {
  if (!l1_indptr || !plan0 || !plan1 || !l0_o_indptr || !l1_o_indptr || !l0_part_rows || !merge_indptr ||
      (l1_batch > 0 && !l1_part_rows) || members < 1 || members > l1_batch || shared_pages < 1 ||
      wave_ctas < 1 || num_kv_heads < 1 || num_qo_heads < num_kv_heads || num_qo_heads % num_kv_heads != 0 ||
      num_qo_heads > INT32_MAX / members)
    return PA_EINVAL;
  if (l1_indptr[0] != 0) return PA_EGEOMETRY;
  // member m's request in the level-1 table: distinct, in range
  std::vector<int32_t> member_of(l1_batch, -1), req_of(members);
  for (int32_t m = 0; m < members; ++m) {
    const int32_t r = member_requests ? member_requests[m] : m;
    if (r < 0 || r >= l1_batch || member_of[r] >= 0) return PA_EINVAL;
    member_of[r] = m;
    req_of[m] = r;
  }
  const int32_t group = num_qo_heads / num_kv_heads;
  const int32_t hpc0 = pa_v2_q_heads_per_cta(members * group, head_dim, kv_dtype);
  const int32_t hpc1 = pa_v2_q_heads_per_cta(group, head_dim, kv_dtype);
  if (hpc0 == 0 || hpc1 == 0) return PA_EUNSUPPORTED;
  const int64_t per0 = static_cast<int64_t>(num_kv_heads) * ((members * group + hpc0 - 1) / hpc0);
  const int64_t per1 = static_cast<int64_t>(num_kv_heads) * ((group + hpc1 - 1) / hpc1);
  std::vector<int64_t> pages1(l1_batch);
  int64_t longest = shared_pages;
  for (int32_t r = 0; r < l1_batch; ++r) {
    pages1[r] = static_cast<int64_t>(l1_indptr[r + 1]) - l1_indptr[r];
    if (pages1[r] < 0) return PA_EGEOMETRY;
    longest = std::max(longest, pages1[r]);
  }
  // a common chunk size for both levels: the smallest whose CTAs (non-increasing in the size) fit the wave
  auto ctas = [&](int64_t size) {
    int64_t n = per0 * ((shared_pages + size - 1) / size);
    for (int64_t p : pages1) n += per1 * (p > size ? (p + size - 1) / size : 1);
    return n;
  };
  int64_t lo = 1, hi = longest;
  if (ctas(hi) > wave_ctas) {
    lo = hi;
  } else {
    while (lo < hi) {
      const int64_t mid = lo + (hi - lo) / 2;
      if (ctas(mid) <= wave_ctas) hi = mid; else lo = mid + 1;
    }
  }
  const int32_t ppc = static_cast<int32_t>(lo);
  // Level 0 then takes the CTAs that size leaves idle: its chunks carry the members' stacked query heads
  // (members x G per KV head against level 1's G), so its pages cost the most; its size is the smallest
  // whose chunks fit the wave beside level 1's chunks at the common size (it only shrinks).
  int32_t ppc0 = ppc;
  if (ctas(lo) <= wave_ctas) {
    int64_t n1 = 0;
    for (int64_t p : pages1) n1 += per1 * (p > lo ? (p + lo - 1) / lo : 1);
    const int64_t chunks0 = std::min<int64_t>((wave_ctas - n1) / per0, PA_V2_MAX_CHUNKS);  // >= ceil(shared / lo)
    ppc0 = static_cast<int32_t>((shared_pages + chunks0 - 1) / chunks0);
  }

  const int32_t ip0[2] = {0, shared_pages};
  const int32_t lp0[1] = {page_size};
  const int32_t fp0[1] = {0};
  pa_status rc = pa_v2_plan(ip0, lp0, fp0, nullptr, 1, page_size, members * num_qo_heads, num_kv_heads, head_dim,
                            kv_dtype, wave_ctas, ppc0, l0_request_indices, l0_kv_tile_indices, l0_cap_chunks,
                            l0_o_indptr, plan0);
  if (rc != PA_OK) return rc;
  plan0->stack_members = members;
  rc = pa_v2_plan(l1_indptr, l1_last_page_len, l1_first_page_offset, l1_seq_lens, l1_batch, page_size,
                  num_qo_heads, num_kv_heads, head_dim, kv_dtype, wave_ctas, ppc, l1_request_indices,
                  l1_kv_tile_indices, l1_cap_chunks, l1_o_indptr, plan1);
  if (rc != PA_OK) return rc;

  // merge input: request r's rows are its level-0 chunks (members), then its level-1 chunks
  const int32_t n0 = plan0->num_chunks;
  int32_t row = 0;
  for (int32_t r = 0; r < l1_batch; ++r) {
    merge_indptr[r] = row;
    const int32_t first1 = l1_o_indptr[r];
    if (member_of[r] >= 0) {
      l0_part_rows[member_of[r]] = row;
      row += n0;
    }
    l1_part_rows[r] = row - first1;  // chunk j of request r (o_indptr[r] <= j) lands at row + j - first1
    row += l1_o_indptr[r + 1] - first1;
  }
  merge_indptr[l1_batch] = row;
  return PA_OK;
}
