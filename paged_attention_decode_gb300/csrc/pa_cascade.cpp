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
