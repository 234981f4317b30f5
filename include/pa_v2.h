/*
 * pa_v2.h -- C ABI of libpa_v2.so: fused paged-attention decode v2 on GB300 (sm_103a).
 *
 * Three calls make one decode step, as the problem statement lays them out
 * (issue #898 "Fused paged-attention decode v2: CSR page table, cross-CTA
 * split-KV, and variable-length merge kernels", design pieces 1-4 and Task
 * 2-4; PR #984 "fused paged-attention decode v2 with CSR page table and
 * cross-CTA split-KV", What changed 2-5):
 *
 *   pa_v2_plan            host: validate the CSR geometry, choose the chunk size
 *                         and emit the flat chunk index arrays (plain data,
 *                         reusable across steps).
 *   pa_v2_decode_partial  device: one CTA per (chunk, kv head, q-head group)
 *                         writes each chunk's normalized partial output and
 *                         its base-2 log-sum-exp.
 *   pa_merge_states       device: variable-length merge of (V, LSE) rows grouped
 *                         by o_indptr.  Skipped when plan.needs_merge == 0: the
 *                         partial output is then already the answer.
 *
 * Conventions for every call:
 *  - Ownership.  The library allocates no device memory and keeps no pointer
 *    after a call returns.  Every buffer belongs to the caller; the plan
 *    states the partial-workspace sizes up front.
 *  - Errors.  Calls return a pa_status; nothing is printed and nothing is
 *    thrown.  Arguments are validated on the host before any launch; a
 *    rejected call launches nothing.  Launch failures return PA_ECUDA.
 *  - Device-side checks.  Device index arrays cannot be validated on the
 *    host.  The kernels bounds-check every page slot, page id and o_indptr
 *    entry they read; an out-of-range value is skipped (its loads are not
 *    issued) and, when the caller passes a status word, recorded there by
 *    OR-ing PA_DEVICE_* bits.  The status word is read by the caller after
 *    the stream has synchronized.
 *  - Streams.  Device calls are asynchronous on the given cudaStream_t
 *    (passed as void*; NULL is the legacy default stream).  Every kernel is
 *    launched with programmatic stream serialization: it may become resident
 *    while the kernel before it in the stream is finishing, but it waits for
 *    that kernel to complete (griddepcontrol.wait) before any global-memory
 *    access that reaches its results, so stream order is kept for every
 *    buffer.  (Before that wait, the partial kernels of a one-request plan
 *    read their first page ids through L2 and prefetch those K/V rows into
 *    L2: speculative reads, range-checked, never written and never used for
 *    a result, which is computed from what is read after the wait.)  Each
 *    kernel also lets the one after it be scheduled early, at its own start.
 *  - Units.  Every LSE is in log2 units (scores run in base 2 with log2(e)
 *    folded into the scale); the natural-log LSE is lse2 * ln 2.
 *  - Layouts are row-major and contiguous:
 *      q            [batch, num_qo_heads, head_dim]              float32
 *      k_pool/v_pool [num_pages, page_size, num_kv_heads, head_dim] kv_dtype
 *      indices      [indptr[batch]] int32 physical page ids
 *      indptr       [batch + 1]     int32 prefix sums of pages per request
 *      last_page_len, first_page_offset [batch] int32
 *    Query head h reads KV head h / (num_qo_heads / num_kv_heads).
 */
#ifndef PA_V2_H
#define PA_V2_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_EINVAL = -1,        /* a null pointer, a negative size or a misaligned buffer */
    PA_EGEOMETRY = -2,     /* the CSR page table breaks the geometry rules */
    PA_ECAPACITY = -3,     /* caller's chunk arrays too small; plan->num_chunks holds the need */
    PA_EUNSUPPORTED = -4,  /* a head_dim / dtype / page_size the kernels do not serve */
    PA_ECUDA = -5,         /* a CUDA runtime call or a launch failed */
    PA_EOOB = -6           /* device-side out-of-range data (see pa_status_from_device) */
} pa_status;

typedef enum pa_dtype { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2 } pa_dtype;

/* Device status bits (OR-ed into the optional status word). */
#define PA_DEVICE_BAD_REQUEST   0x1  /* request_indices entry outside [0, batch) */
#define PA_DEVICE_BAD_SLOT      0x2  /* a page slot outside [0, num_indices) */
#define PA_DEVICE_BAD_PAGE      0x4  /* a page id outside [0, num_pages) */
#define PA_DEVICE_BAD_INDPTR    0x8  /* o_indptr decreasing or outside [0, num_partials] */
#define PA_DEVICE_WAIT_TIMEOUT  0x10 /* a bounded wait (staged K/V, a tensor-memory kernel role) gave up */
#define PA_DEVICE_BAD_BLOCK     0x20 /* a selected block id outside the scored range */

/* Largest chunk count of any plan: the 65535 grid-z bound of the pages'
 * launch shape (PR #984, What changed 4), kept as a plan invariant. */
#define PA_V2_MAX_CHUNKS 65535

/* The plan (PR #984, What changed 4; issue #898, design piece 4).  Plain old
 * data: it can be copied, cached and reused across decode steps for as long
 * as pa_v2_plan_matches() holds, i.e. until a request crosses a page
 * boundary.  Chunk c covers page slots [t * pages_per_chunk,
 * min((t + 1) * pages_per_chunk, pages_r)) of request r =
 * request_indices[c], t = kv_tile_indices[c]; chunks are in request order. */
typedef struct pa_v2_plan_t {
    int32_t batch, num_qo_heads, num_kv_heads, head_dim, page_size;
    int32_t kv_dtype;                 /* pa_dtype */
    int32_t q_heads_per_cta, q_groups;
    int32_t pages_per_chunk;          /* chosen chunk size in pages */
    int32_t lo_pages_per_chunk;       /* smallest launchable size (chunk-count floor) */
    int32_t hi_pages_per_chunk;       /* max(1, longest request in pages) */
    int32_t num_chunks;               /* N: rows of the partial workspace */
    int32_t needs_merge;              /* 1 iff num_chunks > batch */
    int32_t target_ctas, total_ctas;  /* total_ctas = num_chunks * num_kv_heads * q_groups */
    int32_t kernel;                   /* 0: tensor cores for f16/bf16 pools, CUDA cores for f32;
                                         1: CUDA cores (needs q_heads_per_cta <= 8 for head_dim
                                         64 / 128); 2 (head_dim 512 only): the warp-level
                                         tensor-core kernel.  Set by the caller after pa_v2_plan;
                                         pa_v2_plan writes 0. */
    int32_t stack_members;            /* Cascade level 0 (cascade-attention.md): when M > 1 the plan's
                                         single request holds the query heads of M members stacked
                                         h0 = kv*(M*Gm) + m*Gm + g (Gm = num_qo_heads / (M *
                                         num_kv_heads)); q is read, and pa_v2_decode's out / lse2 are
                                         written, in member layout [M, Hm, D] / [M, Hm].  Set by the
                                         caller; pa_v2_plan writes 1. */
    int32_t out_row_step;             /* pa_v2_decode writes final row r (request, or member when
                                         stacked) at row r * out_row_step of out / lse2, so two
                                         decodes can fill interleaved rows for one pa_merge_states.
                                         pa_v2_plan writes 1. */
    int64_t num_indices;              /* indptr[batch] */
    int64_t workspace_v_bytes;        /* num_chunks * num_qo_heads * head_dim * 4 */
    int64_t workspace_lse_bytes;      /* num_chunks * num_qo_heads * 4 */
    int64_t counter_bytes;            /* batch * num_kv_heads * q_groups * 4 (pa_v2_decode) */
    uint64_t geometry_hash;           /* FNV-1a of batch and per-request page counts */
} pa_v2_plan_t;

/* Query heads one CTA serves for GQA group size `group_size`: up to 16 for
 * f16/bf16 pools (tensor-core kernel), up to 8 for f32 pools (CUDA-core
 * kernel); head_dim 512 (the second-K-stream kernels, f16/bf16) up to 32, the
 * tensor-memory kernel's N.  The plan and the launcher both call this, so the
 * CTA count and the grid cannot drift apart (PR #984, What changed 2).
 * Returns 0 for an unsupported shape. */
int32_t pa_v2_q_heads_per_cta(int32_t group_size, int32_t head_dim, int32_t kv_dtype);

/* Occupancy-derived CTA target for `device`: SM count times the partial
 * kernel's resident CTAs per SM for this shape (issue #898, Task 4: "a target
 * derived from SM count").  Writes *target_ctas. */
pa_status pa_v2_default_target_ctas(int32_t device, int32_t num_qo_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t page_size, int32_t kv_dtype,
                                    int32_t* target_ctas);

/* Build a plan.  All pointers are HOST pointers.
 *  indptr [batch+1], last_page_len [batch], first_page_offset [batch]: the CSR
 *    geometry.  Checked: indptr[0] == 0 and non-decreasing; a request with
 *    pages has 1 <= last_page_len <= page_size, 0 <= first_page_offset <
 *    page_size, and first_page_offset < last_page_len when it has one page; a
 *    request with no pages has last_page_len == first_page_offset == 0.
 *  seq_lens [batch] (nullable): when given, the identity
 *    (pages-1)*page_size + last_page_len - first_page_offset == seq_len is
 *    checked for every request (PR #984, What changed 1).
 *  target_ctas > 0: the CTA count to reach; pages_per_chunk_override > 0
 *    fixes the chunk size instead of searching.
 *  request_indices / kv_tile_indices [cap_chunks], o_indptr [batch+1]: outputs.
 * Returns PA_EGEOMETRY on a bad table, PA_EUNSUPPORTED for a shape the
 * kernels do not serve, PA_EINVAL when no chunk size keeps the chunk count
 * within PA_V2_MAX_CHUNKS, and PA_ECAPACITY (with out->num_chunks set) when
 * cap_chunks is too small.  Always sufficient: cap_chunks >=
 * sum_r max(1, pages_r). */
pa_status pa_v2_plan(const int32_t* indptr, const int32_t* last_page_len,
                     const int32_t* first_page_offset, const int32_t* seq_lens, int32_t batch,
                     int32_t page_size, int32_t num_qo_heads, int32_t num_kv_heads,
                     int32_t head_dim, int32_t kv_dtype, int32_t target_ctas,
                     int32_t pages_per_chunk_override, int32_t* request_indices,
                     int32_t* kv_tile_indices, int32_t cap_chunks, int32_t* o_indptr,
                     pa_v2_plan_t* out);

/* The smallest pages_per_chunk whose CTA count -- sum over requests of
 * max(1, ceil(pages_r / ppc)) * ctas_per_chunk, pages_r = indptr[r+1] -
 * indptr[r] -- is at most `wave`; pass it to pa_v2_plan as
 * pages_per_chunk_override.  pa_v2_plan's own search takes the largest size
 * that still reaches its target, so its CTA count can pass one wave (one CTA
 * per SM) by up to a chunk per request.  Returns the one-chunk-per-request
 * size when even that does not fit, 0 for bad arguments.  Host pointers;
 * ctas_per_chunk = num_kv_heads * q_groups of the plan. */
int32_t pa_v2_wave_fit_pages_per_chunk(const int32_t* indptr, int32_t batch, int32_t ctas_per_chunk,
                                       int32_t wave);

/* A pages_per_chunk at or below `pages_per_chunk` (normally the plan's own
 * choice) with the same chunk count -- sum over requests of
 * max(1, ceil(pages_r / ppc)) -- whose chunks give each of the 8 warps of the
 * tensor-core partial kernel the same number of stages (a stage is 16 pool
 * rows: floor(16 / page_size) pages, or a 16-row slice of a page when
 * page_size is a multiple of 16); the largest such size, else
 * `pages_per_chunk` itself (also for page sizes above 16 that are not
 * multiples of 16).  A launch ends with its busiest warp: at 32768 tokens of
 * 16-row pages, 112 pages per chunk (14 stages per warp) against the search's
 * 113 (one warp with 15).  Pass the result to pa_v2_plan as
 * pages_per_chunk_override.  0 for bad arguments.  Host pointers. */
int32_t pa_v2_balanced_pages_per_chunk(const int32_t* indptr, int32_t batch, int32_t page_size,
                                       int32_t pages_per_chunk);

/* 1 if `plan` is still valid for this geometry (same batch and per-request
 * page counts, and a geometry that passes the checks of pa_v2_plan); else 0.
 * Host pointers. */
int32_t pa_v2_plan_matches(const pa_v2_plan_t* plan, const int32_t* indptr,
                           const int32_t* last_page_len, const int32_t* first_page_offset,
                           int32_t batch);

/* The partial kernel (issue #898, design piece 2 and Task 2; PR #984, What
 * changed 2).  One CTA per (chunk, kv head, q-head group) walks the chunk's
 * pages through the CSR table, reads every K/V element once for all query
 * heads of its group, runs an online softmax in base 2 in f32 and writes
 *   v_out   [num_chunks, num_qo_heads, head_dim] f32: the chunk's normalized output
 *   lse2_out [num_chunks, num_qo_heads]          f32: its log2-LSE
 * An empty chunk (a request with no visible token) writes zeros and -inf.
 * When plan->needs_merge == 0 these rows are the final output, one per
 * request.  All array pointers are DEVICE pointers; `plan` is a host pointer.
 * Alignment: pools, q, v_out 16-byte aligned.  num_pages: pool pages
 * (num_pages * page_size < 2^31).  num_indices: length of `indices`.
 * status: nullable device int32 receiving PA_DEVICE_* bits.
 * A one-request plan (batch 1) given num_indices == plan->num_indices fixes
 * chunk c to tile c of request 0 over page slots 0 .. num_indices-1, so the
 * kernel reads neither request_indices / kv_tile_indices nor indptr (they
 * must still be the plan's; pa_v2_plan_matches checks a host indptr).
 * Supported: head_dim 64 or 128; kv_dtype f32, f16, bf16; page_size 1..16 or
 * a multiple of 16 up to 256 (head_dim 512 plans: pa_v2_decode_partial_extra). */
pa_status pa_v2_decode_partial(const pa_v2_plan_t* plan, const float* q, const void* k_pool,
                               const void* v_pool, int32_t kv_dtype, int64_t num_pages,
                               const int32_t* indices, int64_t num_indices, const int32_t* indptr,
                               const int32_t* last_page_len, const int32_t* first_page_offset,
                               const int32_t* request_indices, const int32_t* kv_tile_indices,
                               float sm_scale, float* v_out, float* lse2_out, int32_t* status,
                               void* cuda_stream);

/* One-launch decode step: the partial kernel above with the merge of
 * pa_merge_states fused into it (the "write O directly" single-chunk case and
 * the multi-chunk merge of issue #898, Task 2-3, in one kernel).  Every CTA
 * writes its chunk's partial to the workspace and takes a ticket on the
 * counter of its (request, kv head, q-head group); the CTA holding the last
 * ticket merges all chunks of that request for its heads (closed form of
 * design piece 3) into out / lse2_out and sets the counter back to 0.  No CTA
 * ever waits for another.  A request with one chunk is written straight to
 * out.  Results equal pa_v2_decode_partial + pa_merge_states up to f32
 * rounding order.
 *   o_indptr      [batch + 1] device, the plan's o_indptr
 *   workspace_v / workspace_lse: as v_out / lse2_out of pa_v2_decode_partial
 *   counters      [plan->counter_bytes / 4] device int32, ALL ZERO before the
 *                 first call; the kernel leaves them zero.  After a call that
 *                 failed on the device (status word non-zero), zero them again.
 *   out [batch, num_qo_heads, head_dim] f32, lse2_out [batch, num_qo_heads] f32.
 *   member_rows   nullable device int32 [stack_members]: for a stacked plan,
 *                 the q row group (request) of member m; null means m.
 *   out_rows      nullable device int32 [batch, or stack_members when stacked]:
 *                 the row of out / lse2 that request (member) r is written to;
 *                 null means r * plan->out_row_step.  (pa_v2_cascade_split
 *                 produces both maps for a mixed cascade batch.)
 * Other arguments, layouts and errors as pa_v2_decode_partial.  Two calls
 * sharing `counters` must not overlap on the GPU. */
pa_status pa_v2_decode(const pa_v2_plan_t* plan, const float* q, const void* k_pool, const void* v_pool,
                       int32_t kv_dtype, int64_t num_pages, const int32_t* indices, int64_t num_indices,
                       const int32_t* indptr, const int32_t* last_page_len, const int32_t* first_page_offset,
                       const int32_t* request_indices, const int32_t* kv_tile_indices, const int32_t* o_indptr,
                       float sm_scale, float* workspace_v, float* workspace_lse, int32_t* counters, float* out,
                       float* lse2_out, const int32_t* member_rows, const int32_t* out_rows, int32_t* status,
                       void* cuda_stream);

/* Shared-prefix detection for cascade decode (cascade-attention.md, the
 * detection paragraphs and their table).  Requests with first_page_offset != 0
 * or fewer than 2 pages are left out; the rest are grouped by their first page
 * id; a group's shared span is the number of leading page positions on which
 * all members hold the same page id, capped at pages - 1 for every member; the
 * group with the largest shared * (members - 1) wins (ties: the group whose
 * first member comes first).  It is reported only with at least
 * max(2, min_members) members and min_shared_pages shared pages; otherwise
 * *num_members = 0.  HOST pointers: indptr [batch+1], indices [indptr[batch]],
 * first_page_offset [batch]; member_of [batch] receives 1 for members, 0 else. */
pa_status pa_v2_cascade_detect(const int32_t* indptr, const int32_t* indices,
                               const int32_t* first_page_offset, int32_t batch,
                               int32_t min_shared_pages, int32_t min_members, int32_t* member_of,
                               int32_t* num_members, int32_t* shared_pages);

/* Split a batch into the two cascade levels (cascade-attention.md).  Level 0
 * is the first `shared_pages` pages of the members (all full), attended once
 * with the members' heads stacked; level 1 is every request's remaining pages
 * (members: after the shared span; others: all of them).  The merge input has
 * one row group per request: members two rows (level 0 first, level 1 second),
 * others one row.  HOST pointers.  Outputs: l1_indptr [batch+1], l1_indices
 * [indptr[batch] - members * shared_pages], l1_last_page_len / l1_first_page_offset
 * [batch], member_rows [members] (request of member m, batch order),
 * l0_out_rows [members] and l1_out_rows [batch] (merge-input rows written by
 * level 0 / level 1, for pa_v2_decode's out_rows), merge_indptr [batch+1]. */
pa_status pa_v2_cascade_split(const int32_t* indptr, const int32_t* indices, const int32_t* last_page_len,
                              const int32_t* first_page_offset, int32_t batch, const int32_t* member_of,
                              int32_t shared_pages, int32_t* l1_indptr, int32_t* l1_indices,
                              int32_t* l1_last_page_len, int32_t* l1_first_page_offset,
                              int32_t* member_rows, int32_t* l0_out_rows, int32_t* l1_out_rows,
                              int32_t* merge_indptr);

/* Plans of the two cascade levels (cascade-attention.md, composition and
 * head-stacking paragraphs) for ONE launch of both (pa_v2_cascade_decode),
 * and the layout of the merge input they share.
 *  - Level 0: the `shared_pages` full pages shared by `members` requests, as
 *    one request whose members' query heads are stacked (stack_members =
 *    members, num_qo_heads = members * num_qo_heads).
 *  - Level 1: every request's own table (l1_indptr, l1_last_page_len,
 *    l1_first_page_offset, l1_seq_lens or null; l1_batch requests, host
 *    arrays as for pa_v2_plan).  member_requests[m] (host, or null for m) is
 *    member m's request in that table.
 * Chunk sizes: first the common size, the smallest whose CTAs -- one chunk's
 * CTAs (num_kv_heads x q-groups of the level) per chunk, summed over both
 * levels -- fit `wave_ctas` (the longest request's size when none fits);
 * level 1 takes it.  Level 0, whose chunks carry the stacked heads of every
 * member, takes the CTAs left over: the smallest size whose chunks fit
 * `wave_ctas` beside level 1's (at most the common size; when nothing fits,
 * the common size).  No CTA of the launch reads more pages than the common
 * size.  Each plan
 * is written as pa_v2_plan writes it (arrays into the l0_ / l1_ buffers;
 * level 0 has one request, so l0_o_indptr holds 2 entries), plan0 with
 * stack_members = members.  The merge input puts request r's rows together:
 * its level-0 chunks (members only), then its level-1 chunks.
 *   merge_indptr [l1_batch + 1] (host): request r's first row; the total,
 *     merge_indptr[l1_batch], is the rows of merge_v / merge_lse;
 *   l0_part_rows [members], l1_part_rows [l1_batch] (host): chunk c of
 *     member m (level 0) / of request r (level 1, c its index among level 1's
 *     chunks) goes to row part_rows[m or r] + c.
 * Errors: PA_EINVAL (null pointers, members < 1 or > l1_batch, shared_pages
 * < 1, wave_ctas < 1, a member_requests entry outside [0, l1_batch) or
 * repeated), PA_EGEOMETRY, the errors of pa_v2_plan (PA_ECAPACITY with the
 * plan's num_chunks filled in when a level's arrays are too small). */
pa_status pa_v2_cascade_plan(int32_t members, int32_t shared_pages, const int32_t* l1_indptr,
                             const int32_t* l1_last_page_len, const int32_t* l1_first_page_offset,
                             const int32_t* l1_seq_lens, int32_t l1_batch, const int32_t* member_requests,
                             int32_t page_size, int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t kv_dtype, int32_t wave_ctas, int32_t* l0_request_indices,
                             int32_t* l0_kv_tile_indices, int32_t l0_cap_chunks, int32_t* l0_o_indptr,
                             int32_t* l1_request_indices, int32_t* l1_kv_tile_indices, int32_t l1_cap_chunks,
                             int32_t* l1_o_indptr, int32_t* l0_part_rows, int32_t* l1_part_rows,
                             int32_t* merge_indptr, pa_v2_plan_t* plan0, pa_v2_plan_t* plan1);

/* One cascade level's device arrays for pa_v2_cascade_decode: its page table
 * and plan arrays, member_rows (level 0 of a stacked plan: the q row group of
 * member m, or null for m) and part_rows: the merge-input row of the level's
 * first chunk of each request (member, for level 0), so that chunk c of
 * request r lands in row part_rows[r] + c (pa_v2_cascade_plan computes both
 * levels' part_rows; a row at or past merge_rows is not written and sets
 * PA_DEVICE_BAD_INDPTR in the status word).  DEVICE pointers, owned by the
 * caller. */
typedef struct pa_v2_cascade_level_t {
    const int32_t* indices;
    int64_t num_indices;
    const int32_t* indptr;
    const int32_t* last_page_len;
    const int32_t* first_page_offset;
    const int32_t* request_indices;
    const int32_t* kv_tile_indices;
    const int32_t* member_rows;
    const int32_t* part_rows;
} pa_v2_cascade_level_t;

/* Cascade decode in two launches (cascade-attention.md, composition
 * paragraphs: each request's softmax states over the shared span and over its
 * own pages merge with the closed form of the split-KV merge, which is
 * associative).  ONE launch of the tensor-core partial kernel runs both
 * levels' chunks -- CTAs [0, plan0->num_chunks) level 0, the rest level 1 --
 * and writes every chunk's normalized partial and lse2 into row
 * part_rows[r] + c of merge_v [merge_rows, num_qo_heads, D] / merge_lse
 * [merge_rows, num_qo_heads] (level 0 in member head layout); then
 * pa_merge_states folds rows merge_indptr[r] .. merge_indptr[r + 1] - 1 into
 * out [batch_out, num_qo_heads, D] / lse2_out [batch_out, num_qo_heads].
 * With pa_v2_cascade_plan's part_rows and merge_indptr, request r's rows are
 * its level-0 chunks (members only) followed by its level-1 chunks.  The two
 * plans must share kv_dtype, head_dim, page_size and num_kv_heads, level 0's
 * query heads must be level 1's times its stack_members, and both must take
 * the tensor-core kernel with the same staging (else PA_EUNSUPPORTED); a
 * level without chunks is PA_EINVAL.  q, the
 * pools and num_pages are shared; level 0 reads q through its stacked plan.
 * DEVICE pointers; stream ordered; errors as pa_v2_decode_partial and
 * pa_merge_states. */
pa_status pa_v2_cascade_decode(const pa_v2_plan_t* plan0, const pa_v2_plan_t* plan1,
                               const pa_v2_cascade_level_t* level0, const pa_v2_cascade_level_t* level1,
                               const float* q, const void* k_pool, const void* v_pool, int32_t kv_dtype,
                               int64_t num_pages, float sm_scale, float* merge_v, float* merge_lse,
                               int32_t merge_rows, const int32_t* merge_indptr, int32_t batch_out, float* out,
                               float* lse2_out, int32_t* status, void* cuda_stream);

/* Partial attention with a second K stream (sparse-paged-decode.md, issue
 * #904: the DSA paragraphs, third way out -- "a row stride plus a second K
 * stream").  The score of visible token t (resolved through the page table
 * exactly as in pa_v2_decode_partial) for query head h of kv head kvh is
 *   scale * (q[h] . K_t[0:Dim]) + scale * (q_extra[h] . E_t[0:ExtraDim])
 * and the output is the softmax-weighted sum of V_t[0:Dim], with
 *   K_t = k_pool       + ((page*page_size + e) * num_kv_heads + kvh) * k_row_stride
 *   E_t = k_extra_pool + (same row) * k_extra_row_stride
 *   V_t = v_pool       + (same row) * v_row_stride      (elements of kv_dtype)
 * Row strides (RowStride) may exceed the dims read: the DSA K buffer holds
 * concat(kv_latent, indexer_key) per row and only the latent part is a key.
 * For MLA the values are the latent rows: pass v_pool == k_pool with the same
 * stride and each row is read once.  Kernels, by plan->kernel:
 *   0 (default) values in the key tile (v_pool == k_pool, same stride): the
 *     tensor-memory kernel -- tcgen05.mma, M=128 rows x N=64, accumulators in
 *     tensor memory, up to 32 query heads per CTA; separate values: as 2.
 *   1 CUDA cores, f32 arithmetic, 8 query heads per CTA.
 *   2 warp-level tensor cores (mma.sync m16n8k16), 8 query heads per CTA.
 * Every tensor-core path splits q and P into hi + lo 16-bit halves and
 * accumulates in f32.  The 8-head kernels regroup the plan's query heads at
 * launch; the plan's chunks are used as they are.
 *   plan        from pa_v2_plan with head_dim = Dim = 512 (up to 32 query heads
 *               per CTA, pa_v2_q_heads_per_cta); stack_members and
 *               out_row_step 1; kernel 0, 1 or 2 (else PA_EINVAL).
 * A one-request plan given num_indices == plan->num_indices reads no chunk
 * arrays or indptr, as in pa_v2_decode_partial.
 *   q [batch, num_qo_heads, 512] f32 (16-byte aligned), q_extra [batch,
 *   num_qo_heads, 64] f32 (8-byte aligned).
 *   extra_dim   must be 64 (ExtraDim).
 *   strides     in elements, multiples of 8, k/v >= 512, extra >= 64; pools
 *               16-byte aligned.
 *   v_out [num_chunks, num_qo_heads, 512] f32 (16-byte aligned) and lse2_out
 *   [num_chunks, num_qo_heads] f32 as pa_v2_decode_partial; pa_merge_states
 *   combines them.
 * kv_dtype f16 or bf16.  Other arguments, device checks and errors as
 * pa_v2_decode_partial; PA_EUNSUPPORTED for other dims or dtypes. */
pa_status pa_v2_decode_partial_extra(const pa_v2_plan_t* plan, const float* q, const float* q_extra,
                                     const void* k_pool, int64_t k_row_stride, const void* v_pool,
                                     int64_t v_row_stride, const void* k_extra_pool, int64_t k_extra_row_stride,
                                     int32_t extra_dim, int32_t kv_dtype, int64_t num_pages,
                                     const int32_t* indices, int64_t num_indices, const int32_t* indptr,
                                     const int32_t* last_page_len, const int32_t* first_page_offset,
                                     const int32_t* request_indices, const int32_t* kv_tile_indices,
                                     float sm_scale, float* v_out, float* lse2_out, int32_t* status,
                                     void* cuda_stream);

/* Self-test of the tensor-memory kernel's bounded waits, for failure-detection
 * tests (no tensor memory, no copies, one CTA of 2 warps): warp 0 waits on an
 * mbarrier nothing arrives on for about limit_cycles SM clocks, gives up,
 * records PA_DEVICE_WAIT_TIMEOUT in *status and raises the CTA's abort flag;
 * warp 1 waits on another with the kernels' full limit (about 2^31 cycles) and
 * must give up through that flag.  completed[2] (device int32) receives 1 for a
 * warp whose wait completed (neither may).  status, completed: DEVICE pointers.
 * PA_EINVAL for limit_cycles outside [1024, 2^31]. */
pa_status pa_v2_selftest_wait(int32_t* status, int32_t* completed, int64_t limit_cycles, void* cuda_stream);

/* Block-sparse selections (sparse-paged-decode.md, issue #904: the paragraphs
 * on selection_from_blocks and on the final block).  A model that scores
 * blocks of `block_size` positions picks `topk` of the blocks 0 .. nb-2 of
 * each request, nb = ceil(kv_len / block_size); the final block nb-1 (the
 * query's own) is never scored and is always attended, its live
 * kv_len - (nb-1)*block_size rows only.  The count of rows per request,
 *   per_request = topk * block_size + kv_len - (nb-1)*block_size,
 * depends on kv_len alone, so the page table's structure is host data while
 * the rows themselves stay on the device.
 *
 * pa_selection_rows_per_request: per_request, or -1 when the arguments are
 * invalid (block_size < 1, kv_len < 1, topk < 0 or topk > nb - 1). */
int64_t pa_selection_rows_per_request(int32_t topk, int32_t block_size, int32_t kv_len);

/* The page_size-1 CSR structure of a token-exact selection: indptr[r] =
 * r * per_request, last_page_len[r] = 1 (0 when per_request is 0),
 * first_page_offset[r] = 0.  HOST pointers: indptr [num_requests + 1],
 * last_page_len and first_page_offset [num_requests].  PA_EINVAL for negative
 * sizes, null pointers or num_requests * per_request above INT32_MAX. */
pa_status pa_sparse_csr(int32_t num_requests, int64_t per_request, int32_t* indptr, int32_t* last_page_len,
                        int32_t* first_page_offset);

/* Expand the selected block ids into token rows, one device pass over the
 * selected rows (O(selected)): request r's rows are, for each selected block
 * j in the order given, r*request_stride + j*block_size + e for e in
 * [0, block_size), then the final block's live rows
 * r*request_stride + (nb-1)*block_size + e.  With a dense cache
 * [B, H, Cap, D] viewed as the pool [B*H*Cap, 1, 1, D] and requests
 * r = b*H + h, request_stride is the reserved capacity Cap (not the live
 * length).  The result is the `indices` of a page_size-1 decode whose CSR
 * structure pa_sparse_csr gives.
 *   block_ids [num_requests, topk] device int32 (any order, e.g. an
 *             argpartition output); may be null when topk == 0.
 *   indices   [num_requests * per_request] device int32, written.
 * A block id outside [0, nb-1) is not expanded: its rows are written as -1
 * (which the decode kernels reject as a bad page id) and PA_DEVICE_BAD_BLOCK
 * is OR-ed into *status when status is not null.  Host errors: PA_EINVAL for
 * invalid sizes, request_stride < kv_len or a null `indices`; PA_EUNSUPPORTED
 * when a row or the row count does not fit in int32.  Launched like the other
 * kernels (programmatic dependent, asynchronous on cuda_stream). */
pa_status pa_selection_from_blocks(const int32_t* block_ids, int32_t num_requests, int32_t topk,
                                   int32_t block_size, int32_t kv_len, int64_t request_stride,
                                   int32_t* indices, int32_t* status, void* cuda_stream);

/* One whole decode step for callers whose per-step inputs (the query and the
 * page table) are in host memory.  The pages have no counterpart to this call:
 * it packages the step they time (plan built once outside the step; partial,
 * then merge when needs_merge) with the host<->device traffic around it, so
 * that a host-side caller makes one call, one host-to-device copy and one
 * device-to-host copy per step.
 *
 * pa_v2_host_io_layout: byte sizes for a plan.  host_in [in_bytes] holds, as
 * consecutive 4-byte words, q [batch, num_qo_heads, head_dim] f32, indices
 * [num_indices] int32, indptr [batch+1], last_page_len [batch],
 * first_page_offset [batch], then zeros up to in_bytes (the last 16 bytes are
 * the device status slot, zeroed by the copy).  host_out [out_bytes] receives
 * the status word (first 4 bytes of a 16-byte slot), out [batch, num_qo_heads,
 * head_dim] f32 and lse2 [batch, num_qo_heads] f32.  dev_io is a device buffer
 * of io_bytes (16-byte aligned) the call copies into and out of. */
pa_status pa_v2_host_io_layout(const pa_v2_plan_t* plan, int64_t* in_bytes, int64_t* out_bytes,
                               int64_t* io_bytes);

/* pa_v2_decode_host: check that `plan` still matches the page table in host_in
 * (PA_EGEOMETRY if not; nothing is launched), copy host_in to dev_io, run
 * pa_v2_decode_partial (and pa_merge_states when plan->needs_merge, through
 * workspace_v / workspace_lse sized by the plan), copy the status, out and
 * lse2 to host_out, and synchronize `cuda_stream`.  host_in / host_out should
 * be page-locked for the copies to be asynchronous.  k_pool, v_pool, the plan's
 * device arrays (request_indices, kv_tile_indices, o_indptr) and the
 * workspaces are device pointers as for the calls it makes.  Returns the first
 * failing call's status, else pa_status_from_device(status word). */
pa_status pa_v2_decode_host(const pa_v2_plan_t* plan, const void* host_in, void* host_out, void* dev_io,
                            const void* k_pool, const void* v_pool, int32_t kv_dtype, int64_t num_pages,
                            const int32_t* request_indices, const int32_t* kv_tile_indices,
                            const int32_t* o_indptr, float sm_scale, float* workspace_v, float* workspace_lse,
                            void* cuda_stream);

/* pa_v2_decode_host as one CUDA graph, for callers that repeat the step with
 * the same buffers.  create() captures the step (input copy, partial kernel,
 * merge when plan->needs_merge, output copy) into a graph and instantiates it;
 * the plan (copied), host_in, host_out, dev_io, the pools, the chunk arrays,
 * the workspaces and sm_scale are bound then, with the arguments and checks of
 * pa_v2_decode_host.  run() checks the plan against the page table now in
 * host_in (PA_EGEOMETRY, nothing launched), launches the graph on cuda_stream,
 * waits for it and returns pa_status_from_device of the status word, like
 * pa_v2_decode_host; host_in's 16-byte status slot must stay zero.  The bound
 * buffers must outlive the graph; destroy() releases it (null is a no-op).
 * One graph must not run on two streams at once. */
typedef struct pa_v2_host_graph pa_v2_host_graph_t;
pa_status pa_v2_host_graph_create(const pa_v2_plan_t* plan, const void* host_in, void* host_out, void* dev_io,
                                  const void* k_pool, const void* v_pool, int32_t kv_dtype, int64_t num_pages,
                                  const int32_t* request_indices, const int32_t* kv_tile_indices,
                                  const int32_t* o_indptr, float sm_scale, float* workspace_v, float* workspace_lse,
                                  pa_v2_host_graph_t** graph);
pa_status pa_v2_host_graph_run(pa_v2_host_graph_t* graph, void* cuda_stream);
void pa_v2_host_graph_destroy(pa_v2_host_graph_t* graph);

/* The same step with no copies, for a GPU that reaches host memory directly
 * (on a GB300, the Grace CPU's memory over the coherent NVLink-C2C link).
 * host_in and host_out keep the pa_v2_host_io_layout layout but must be
 * page-locked and mapped into the device's address space (cudaHostAlloc, or
 * cudaHostRegister with cudaHostRegisterMapped) and 16-byte aligned; the
 * partial kernel reads q and the page table from host_in through its device
 * address, and the last kernel writes out and lse2 into host_out, whose first
 * 16 bytes are the status slot: the call (or run()) zeroes it from the host
 * before the launch, and the kernels OR their error bits into word 0.  When
 * the plan merges, each merge CTA adds one to word 1 once its results are
 * visible to the host (a system-scope fence first), and the call returns as
 * soon as that count is complete rather than after synchronising cuda_stream
 * (after ~5 s without it, it synchronises): the step's kernels may still be
 * retiring when it returns.  Work queued on cuda_stream afterwards is ordered
 * after them; synchronise the stream before freeing either buffer or handing
 * it to another stream.  host_in's trailing status slot is not used, and
 * there is no dev_io.
 *
 * pa_v2_decode_host_mapped: check the plan against host_in's page table
 * (PA_EGEOMETRY, nothing launched), launch the partial kernel and the merge
 * when plan->needs_merge, wait for the merge's count (or, without a merge,
 * synchronize cuda_stream) and return pa_status_from_device of the status
 * word.  PA_EINVAL as pa_v2_decode_host,
 * and when host_in or host_out is unaligned or has no device mapping.
 *
 * pa_v2_host_graph_create_mapped: capture the same two launches as a graph,
 * bound like pa_v2_host_graph_create; pa_v2_host_graph_run and
 * pa_v2_host_graph_destroy serve both kinds of graph.  Neither host buffer may
 * be written while a step that uses it runs (between the launch and the
 * synchronisation that ends it). */
pa_status pa_v2_decode_host_mapped(const pa_v2_plan_t* plan, const void* host_in, void* host_out, const void* k_pool,
                                   const void* v_pool, int32_t kv_dtype, int64_t num_pages,
                                   const int32_t* request_indices, const int32_t* kv_tile_indices,
                                   const int32_t* o_indptr, float sm_scale, float* workspace_v, float* workspace_lse,
                                   void* cuda_stream);
pa_status pa_v2_host_graph_create_mapped(const pa_v2_plan_t* plan, const void* host_in, void* host_out,
                                         const void* k_pool, const void* v_pool, int32_t kv_dtype, int64_t num_pages,
                                         const int32_t* request_indices, const int32_t* kv_tile_indices,
                                         const int32_t* o_indptr, float sm_scale, float* workspace_v,
                                         float* workspace_lse, pa_v2_host_graph_t** graph);

/* Size of the device scratch array behind pa_v2_decode_noalloc: 8 MiB, held
 * by every GPU that loads this library until the process exits. */
#define PA_V2_NOALLOC_SCRATCH_BYTES (8u << 20)

/* pa_v2_decode for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point; it exists for users whose process
 * does not let them call cudaMalloc: a serving engine that reserves all device
 * memory up front for its own pools, or a plugin that is handed only input and
 * output pointers by its host.  Such a caller cannot provide the partial
 * workspace and ticket counters pa_v2_decode needs, so this call takes them
 * from a fixed array in the library's own device memory
 * (PA_V2_NOALLOC_SCRATCH_BYTES, laid out as counters, then workspace_v, then
 * workspace_lse, each rounded up to 256 bytes).  It allocates nothing.
 *  - The caller still passes every input and output: the same arguments and
 *    layouts as pa_v2_decode, minus workspace_v / workspace_lse / counters
 *    and minus the row maps member_rows / out_rows, which are taken as null:
 *    request r writes output row r * plan->out_row_step, and member m of a
 *    stacked plan reads q row group m and writes row m * plan->out_row_step.
 *  - A plan whose counters plus workspace exceed PA_V2_NOALLOC_SCRATCH_BYTES
 *    is rejected with PA_ECAPACITY before anything is launched.  A plan with
 *    no chunks (batch 0) returns PA_OK and launches nothing.
 *  - The first call on a device looks up that device's copy of the array
 *    (cudaGetSymbolAddress, with that device current) and remembers it for
 *    the life of the process; make that first call before any stream capture.
 *    The remembered address does not survive cudaDeviceReset: do not call
 *    this entry point on a device after resetting it.  If the lookup fails
 *    the call returns PA_ECUDA and clears the runtime's last error.
 *  - Every call on a device shares the one array and leaves its contents
 *    behind.  Each call clears the counter region on its stream
 *    (cudaMemsetAsync) before the launch.  Calls whose work overlaps on the GPU
 *    (different streams, or no ordering between them) race on the array:
 *    order them on one stream. */
pa_status pa_v2_decode_noalloc(const pa_v2_plan_t* plan, const float* q, const void* k_pool,
                               const void* v_pool, int32_t kv_dtype, int64_t num_pages,
                               const int32_t* indices, int64_t num_indices, const int32_t* indptr,
                               const int32_t* last_page_len, const int32_t* first_page_offset,
                               const int32_t* request_indices, const int32_t* kv_tile_indices,
                               const int32_t* o_indptr, float sm_scale, float* out, float* lse2_out,
                               int32_t* status, void* cuda_stream);

/* The variable-length merge (issue #898, design piece 3 and Task 3; PR
 * #984, What changed 3).  For output row r and head h, the rows
 * o_indptr[r] .. o_indptr[r+1]-1 of (v_in, lse2_in) merge by
 *   m = max lse_i, w_i = 2^(lse_i - m),
 *   v_out = sum w_i v_i / sum w_i, lse2_out = log2(sum w_i) + m.
 * A -inf row contributes nothing; a group with no finite row (or no row)
 * gives zeros and -inf.  It knows nothing about paging, so any grouping of
 * contiguous rows works (cascade composition reuses it unchanged).
 *   v_in [num_partials, num_heads, head_dim] f32, lse2_in [num_partials, num_heads] f32,
 *   o_indptr [num_rows_out + 1] int32, v_out [num_rows_out, num_heads, head_dim] f32,
 *   lse2_out [num_rows_out, num_heads] f32.
 * DEVICE pointers; v_in / v_out 16-byte aligned.  status as above. */
pa_status pa_merge_states(const float* v_in, const float* lse2_in, const int32_t* o_indptr,
                          int32_t num_rows_out, int32_t num_partials, int32_t num_heads,
                          int32_t head_dim, float* v_out, float* lse2_out, int32_t* status,
                          void* cuda_stream);

/* Map a device status word (PA_DEVICE_* bits) to a pa_status: 0 -> PA_OK,
 * a wait timeout -> PA_ECUDA, any out-of-range bit -> PA_EOOB. */
pa_status pa_status_from_device(int32_t status_word);

/* Human-readable name of a pa_status value (static storage). */
const char* pa_status_string(int32_t status);

/* Library version string (static storage). */
const char* pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_V2_H */
