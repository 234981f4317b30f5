// pa_partial_extra_tc05.cu -- the second-K-stream partial kernel (MLA / DSA
// decode) on the fifth-generation tensor cores: tcgen05.mma with the
// accumulators in tensor memory.
//
// Contract: as pa_partial_extra.cu (sparse-paged-decode.md, issue #904, the
// DSA paragraphs, third way out):
//   score_t = scale * (q . k[row_t][0:512]) + scale * (q_extra . k_extra[row_t][0:64])
// and the output is the softmax-weighted sum of the latent rows k[row_t][0:512]
// (values read from the key tile: v_pool is k_pool), rows resolved through
// the CSR page table; one CTA per (chunk, kv head, group of up to 32 query
// heads) writes the chunk's normalized partial and its log2-LSE.
//
// Why tensor memory: with every query head on one latent KV head the decode is
// a dense contraction (about 200 flops per byte of K at 128 heads), and the
// O^T tile of 32 heads x 512 dims in f32 (64 KB) lives in tensor memory
// instead of registers, so a CTA serves 32 heads and each K row is read by
// 128 / 32 CTAs instead of 128 / 8.
//
// 288 threads in three roles:
//  - q: one 2 KB bulk copy per head (the copy engine) into the latent blocks the
//    first tile fills last, converted to hi + lo halves by the other 160 threads.
//  - warps 0-3, loaders: gather the chunk's rows 128 at a time with cp.async
//    into a tile of nine 128-byte-swizzled blocks [128 rows x 64 dims] (blocks
//    0-7 the latent dims, block 8 the extra dims), 8 lanes per row and one
//    16-byte chunk per lane; invalid rows are zeroed.  Latent blocks 2j, 2j+1
//    are refilled as soon as the MMAs of O^T m-tile j have completed.
//  - warp 8, MMA: one thread issues, per tile of 128 rows,
//      S^T [128 x 64]  = K [128 x 576] . [Q_hi ; Q_lo]^T      36 MMAs, M=128 N=64
//      O^T [512 x 64] += V^T [512 x 128] . [P_hi ; P_lo]^T     4 x 8 MMAs, M=128 N=64
//    q and P are split into hi + lo halves of the pool's 16-bit type (q with
//    scale*log2(e) folded in); the hi and lo products land in two 32-column
//    halves of S^T and of each O^T m-tile and are added when read.  V^T is the
//    key tile read through an MN-major descriptor; [P_hi ; P_lo]^T sits in the
//    extra-dims block, which S^T has finished with (it is refilled after O^T).
//  - warps 4-7, softmax: thread r owns row r of the tile (tensor-memory lane
//    r); it adds its hi and lo scores, takes the per-head maximum over the 128
//    rows (a warp reduce-scatter plus a 4-warp exchange), writes P^T (hi, lo)
//    to shared memory and keeps per-row partial sums of P.  A head's running
//    maximum is raised only when a tile maximum exceeds it by more than 8
//    (log2 units, so P <= 256); O^T and the partial sums are then rescaled in
//    place.  The result is the same softmax: every term uses one offset per
//    head, and the final LSE adds that offset back.
// At the end the softmax warps reduce the row sums, read O^T out of tensor
// memory and write the chunk's output rows and log2-LSE.
//
// Synchronisation: mbarriers only (no named barriers inside the tile loop);
// every wait is bounded and gives up when another role has given up, so a
// timeout ends the CTA cleanly with PA_DEVICE_WAIT_TIMEOUT in the status word.
// Tensor memory (512 columns) is released by the warp that allocated it after
// all of its MMAs have completed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <type_traits>

#include "pa_internal.cuh"
#include "pa_mma.cuh"

namespace pa {
namespace {

constexpr int kTDim = 512;                  // latent dims (key part and value width)
constexpr int kTExtra = 64;                 // extra dims
constexpr int kTRows = 128;                 // rows per tile (M of S^T)
constexpr int kTHeads = 32;                 // query heads per CTA (N of O^T)
constexpr int kTBlocks = 9;                 // 64-dim blocks of a tile row: 8 latent + 1 extra
constexpr int kTLoadWarps = 4;
constexpr int kTSoftWarp0 = 4;              // softmax warps 4..7 (warp % 4 = tensor-memory lane quarter)
constexpr int kTMmaWarp = 8;
constexpr int kTThreads = 9 * 32;
constexpr int kTLag = 1;                   // copy groups (blocks) in flight behind the newest
constexpr float kTLazy = 8.0f;              // raise a running maximum only past this margin (log2 units)

// shared-memory layout (byte offsets from a 1024-byte-aligned base)
constexpr int kTBlockBytes = kTRows * 128;             // 16 KB: 128 rows x 64 dims
constexpr int kTQBlockBytes = 2 * kTHeads * 128;       // 8 KB: 32 hi rows then 32 lo rows
constexpr int kTPBlockBytes = 2 * kTHeads * 128;       // 8 KB: 32 hi then 32 lo head rows x 64 tokens
constexpr int kTOffK = 0;
constexpr int kTOffP = kTOffK + 8 * kTBlockBytes;          // P^T: the two token halves in the extra block
constexpr int kTOffQ = kTOffK + kTBlocks * kTBlockBytes;   // 147456
constexpr int kTOffRed = kTOffQ + kTBlocks * kTQBlockBytes;  // 221184: [2][4][32] f32
constexpr int kTOffBar = kTOffRed + 2 * 4 * kTHeads * 4;   // 222208
static_assert(2 * kTPBlockBytes == kTBlockBytes, "P^T fills the extra block");
constexpr int kTNumBars = 19;
constexpr int kTOffMisc = kTOffBar + kTNumBars * 8;        // tensor-memory address, abort flag
constexpr int kTSmem = kTOffMisc + 16;
constexpr int kTSmemAlloc = kTSmem + 1024;                 // room to align the base
static_assert(kTSmemAlloc <= 227 * 1024, "shared memory");

// barrier slots
constexpr int kBarFull = 0;      // 9: block b of the tile has landed (128 loader arrivals)
constexpr int kBarS = 9;         // S^T complete (tcgen05.commit)
constexpr int kBarP = 10;        // P^T written, S^T read, O^T rescaled (128 softmax arrivals)
constexpr int kBarPv = 11;       // 4: O^T m-tile j complete (commit): blocks 2j, 2j+1 (and, j = 3, 8) free
constexpr int kBarRed = 15;      // the softmax warps' exchange (128 arrivals)
constexpr int kBarDrain = 16;    // all MMAs complete (commit), before tensor memory is released
constexpr int kBarQ = 17;        // the f32 q rows have landed in the staging area (bulk copies)
constexpr int kBarQc = 18;       // [Q_hi ; Q_lo]^T is written (the 160 non-loader threads)
constexpr int kTQThreads = kTThreads - kTLoadWarps * 32;
constexpr int kTOffQStage = kTOffK + 4 * kTBlockBytes;  // f32 q rows, 32 x 2 KB, in latent blocks 4-7

// tensor-memory columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // S^T: 64 columns (hi heads 0-31, lo heads 0-31)
constexpr uint32_t kColO = 64;   // O^T m-tile j: columns 64 + 64 j (hi heads 0-31, lo heads 0-31)

__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: f32 accumulate, A and B of format fmt
// (0 f16, 1 bf16), A K-major or MN-major, B K-major, M x N.
__host__ __device__ constexpr uint32_t instr_desc(uint32_t fmt, int m, int n, bool a_mn) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((a_mn ? 1u : 0u) << 15) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

#define PA_R32(x)                                                                                         \
  "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), "=r"(x[7]),         \
      "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]), "=r"(x[14]), "=r"(x[15]), \
      "=r"(x[16]), "=r"(x[17]), "=r"(x[18]), "=r"(x[19]), "=r"(x[20]), "=r"(x[21]), "=r"(x[22]),           \
      "=r"(x[23]), "=r"(x[24]), "=r"(x[25]), "=r"(x[26]), "=r"(x[27]), "=r"(x[28]), "=r"(x[29]),           \
      "=r"(x[30]), "=r"(x[31])
#define PA_W32(x)                                                                                          \
  "r"(x[0]), "r"(x[1]), "r"(x[2]), "r"(x[3]), "r"(x[4]), "r"(x[5]), "r"(x[6]), "r"(x[7]), "r"(x[8]),       \
      "r"(x[9]), "r"(x[10]), "r"(x[11]), "r"(x[12]), "r"(x[13]), "r"(x[14]), "r"(x[15]), "r"(x[16]),        \
      "r"(x[17]), "r"(x[18]), "r"(x[19]), "r"(x[20]), "r"(x[21]), "r"(x[22]), "r"(x[23]), "r"(x[24]),       \
      "r"(x[25]), "r"(x[26]), "r"(x[27]), "r"(x[28]), "r"(x[29]), "r"(x[30]), "r"(x[31])
#define PA_REGS32                                                                                     \
  "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26," \
  "%27,%28,%29,%30,%31}"

// 32 consecutive columns of this thread's lane, waited for in the same statement
// so that no use of the registers can be scheduled before the data is there.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 " PA_REGS32 ", [%32];\n\t"
               "tcgen05.wait::ld.sync.aligned;"
               : PA_R32(r)
               : "r"(taddr)
               : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
               "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
               "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
               PA_W32(r)
               : "memory");
}

// One contiguous global -> shared copy on the copy engine, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void cp_async_16_plain(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Warp reduce-scatter over 32 values per lane: afterwards v[0] of lane l is
// the max (or sum) over the warp of entry l.
template <bool MAX>
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool upper = (lane & w) != 0;
#pragma unroll
    for (int k = 0; k < w; ++k) {
      const float keep = upper ? v[k + w] : v[k];
      const float send = upper ? v[k] : v[k + w];
      const float got = __shfl_xor_sync(0xffffffffu, send, w);
      v[k] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  return v[0];
}

// Bounded wait that also gives up once another role has given up (abort flag);
// warp-uniform result.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile uint32_t* abort,
                                           int32_t* status, long long limit = kWaitLimitCycles) {
  bool ok = mbar_try_wait(bar, parity);
  if (!ok) {
    const long long t0 = clock64();
    while (true) {
      if (mbar_try_wait(bar, parity)) {
        ok = true;
        break;
      }
      if (*abort) break;
      if (clock64() - t0 > limit) {
        *abort = 1u;
        report(status, PA_DEVICE_WAIT_TIMEOUT);
        break;
      }
    }
  }
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Row `q` (0-based, in pool rows of the chunk's pages) of chunk geometry g:
// its page slot relative to the request and the entry within the page, and
// whether the row is a visible token.
__device__ __forceinline__ bool chunk_row(const PartialParams& p, const ChunkGeom& g, int q, int* slot, int* e) {
  const int rel = (int)fast_div((uint32_t)q, p.ps_magic, p.ps_shift);
  *slot = g.s_begin + rel;
  *e = q - rel * p.page_size;
  if (*slot >= g.s_end) return false;
  if (*slot == 0 && *e < g.fpo) return false;
  if (*slot == g.pages - 1 && *e >= g.lpl) return false;
  return true;
}

struct Tc05Fields {
  const float* q_extra;
  const void* k_extra;
  int64_t k_stride, e_stride;
};

template <typename T>
__global__ void __launch_bounds__(kTThreads, 1)
    pa_v2_partial_extra_tc05_kernel(const PartialParams p, const Tc05Fields x) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kTOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kTOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + kTOffMisc + 4);
  float* red = reinterpret_cast<float*>(smem + kTOffRed);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int c = blockIdx.x;
  const int kvh = blockIdx.y / p.q_groups;
  const int qg = blockIdx.y % p.q_groups;
  const int h_first = kvh * p.group + qg * p.hpc;
  const int nheads = min(min(p.hpc, kTHeads), p.group - qg * p.hpc);

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int b = 0; b < kTBlocks; ++b) mbar_init(&bars[kBarFull + b], kTLoadWarps * 32);
    mbar_init(&bars[kBarS], 1);
    mbar_init(&bars[kBarP], 128);
    for (int j = 0; j < 4; ++j) mbar_init(&bars[kBarPv + j], 1);
    mbar_init(&bars[kBarRed], 128);
    mbar_init(&bars[kBarDrain], 1);
    mbar_init(&bars[kBarQ], 1);
    mbar_init(&bars[kBarQc], kTQThreads);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == kTMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncwarp();
  __syncthreads();  // barriers initialised, tensor-memory address published
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sbase = smem_addr(smem);
  pdl_wait_prerequisites();

  int r;
  const ChunkGeom gm = chunk_geom(p, c, &r);
  const int rows = gm.n_stages > 0 ? (gm.s_end - gm.s_begin) * p.page_size : 0;
  const int n_tiles = (rows + kTRows - 1) / kTRows;

  // loader state: this thread's 16-byte chunk of its 8 tile rows, and tile 0's page ids (their loads
  // are in flight while the q tile is written)
  const int u = threadIdx.x;
  const int ch = u & 7;
  const int rsub = u >> 3;  // rows rsub + 16 s, s = 0..7
  const T* kpool = static_cast<const T*>(p.k_pool);
  const T* epool = static_cast<const T*>(x.k_extra);
  // pool row of each of this thread's 8 tile rows, or -1 (not a visible token, or a bad page id)
  auto lookup = [&](int i, int64_t (&pr)[8]) {
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      int slot, e;
      pr[s] = -1;
      if (chunk_row(p, gm, i * kTRows + rsub + 16 * s, &slot, &e)) {
        const int32_t page = __ldg(p.indices + gm.slot_base + slot);
        if (page >= 0 && (int64_t)page < p.num_pages)
          pr[s] = ((int64_t)page * p.page_size + e) * p.num_kv_heads + kvh;
        else if (ch == 0)
          report(p.status, PA_DEVICE_BAD_PAGE);
      }
    }
  };
  int64_t prow[8], pnext[8];
  if (warp < kTLoadWarps && n_tiles > 0) lookup(0, pnext);

  // ---- [Q_hi ; Q_lo]^T.  The f32 q rows go to the copy engine (one 2 KB bulk copy per head into
  // latent blocks 4-7, which the first tile does not load until the tile is converted), so they do
  // not queue behind the loaders' row copies; q_extra (8 KB, 8-byte aligned) is read directly.  The
  // 160 non-loader threads convert: block b holds dims 64b .. 64b+63 of 32 hi rows then 32 lo rows.
  bool q_ok = true;
  if (warp >= kTLoadWarps) {
    if (warp == kTMmaWarp) {
      if (lane == 0) mbar_arrive_expect_tx(&bars[kBarQ], (uint32_t)(nheads * kTDim * 4));
      __syncwarp();
      if (lane < nheads)
        bulk_g2s(sbase + kTOffQStage + lane * (kTDim * 4),
                 p.q + ((size_t)r * p.num_qo_heads + h_first + lane) * kTDim, kTDim * 4, &bars[kBarQ]);
    }
    const int tq = threadIdx.x - kTLoadWarps * 32;
    unsigned char* qt = smem + kTOffQ;
    auto put = [&](int h, int d, float a, float b) {  // dims d, d + 1 of head h (d even)
      const float v0 = a * p.scale_log2, v1 = b * p.scale_log2;
      const float h0 = TC<T>::round(v0), h1 = TC<T>::round(v1);
      const int dd = d & 63;
      unsigned char* blk = qt + (d >> 6) * kTQBlockBytes;
      const uint32_t off = sw128(h, dd >> 3) + (dd & 7) * 2;  // rows h and h + 32 share the swizzle phase
      *reinterpret_cast<uint32_t*>(blk + off) = (uint32_t)TC<T>::bits(h0) | ((uint32_t)TC<T>::bits(h1) << 16);
      *reinterpret_cast<uint32_t*>(blk + kTHeads * 128 + off) =
          (uint32_t)TC<T>::bits(v0 - h0) | ((uint32_t)TC<T>::bits(v1 - h1) << 16);
    };
    // q_extra: 32 heads x 32 float2, loads first
    constexpr int kE = kTHeads * (kTExtra / 2);
    constexpr int kEPer = (kE + kTQThreads - 1) / kTQThreads;
    float2 ev[kEPer];
#pragma unroll
    for (int k = 0; k < kEPer; ++k) {
      const int it = tq + k * kTQThreads;
      const int h = it >> 5;
      ev[k] = make_float2(0.f, 0.f);
      if (it < kE && h < nheads)
        ev[k] = __ldg(reinterpret_cast<const float2*>(x.q_extra + ((size_t)r * p.num_qo_heads + h_first + h) * kTExtra +
                                                      (it & 31) * 2));
    }
    q_ok = wait_phase(&bars[kBarQ], 0, abort_flag, p.status);
    if (q_ok) {
      const float* stage = reinterpret_cast<const float*>(smem + kTOffQStage);
      constexpr int kQ4 = kTHeads * (kTDim / 4);  // float4 items
      for (int it = tq; it < kQ4; it += kTQThreads) {
        const int h = it >> 7, d = (it & 127) * 4;
        const float4 v = h < nheads ? *reinterpret_cast<const float4*>(stage + h * kTDim + d)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
        put(h, d, v.x, v.y);
        put(h, d + 2, v.z, v.w);
      }
#pragma unroll
      for (int k = 0; k < kEPer; ++k) {
        const int it = tq + k * kTQThreads;
        if (it < kE) put(it >> 5, kTDim + (it & 31) * 2, ev[k].x, ev[k].y);
      }
    }
    fence_proxy_async_smem();  // the q tile is read by the tensor cores
    mbar_arrive(&bars[kBarQc]);
  }

  if (warp < kTLoadWarps) {
    // ------------------------------------------------------------------ loaders
    bool alive = true;
    for (int i = 0; i < n_tiles && alive; ++i) {
#pragma unroll
      for (int s = 0; s < 8; ++s) prow[s] = pnext[s];
      // one copy group per block, in the order the blocks are freed (latent blocks 2j, 2j+1 once O^T
      // m-tile j of tile i-1 is done, the extra block, which held P^T, with the last pair); block b is
      // published once the groups issued after it leave at most kTLag groups in flight
      // source rows resolved once per tile; the block loop is unrolled, so the 72 copies issue as
      // straight-line code (a loop with per-copy 64-bit address arithmetic issued them at about
      // half the rate, which bounded the kernel)
      const T* ksrc[8];
      const T* esrc[8];
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int64_t pr = prow[s] >= 0 ? prow[s] : 0;
        ksrc[s] = kpool + pr * x.k_stride + ch * 8;
        esrc[s] = epool + pr * x.e_stride + ch * 8;
      }
#pragma unroll
      for (int b = 0; b < kTBlocks; ++b) {
        if (i > 0 && (b & 1) == 0 && b < 8 &&
            !wait_phase(&bars[kBarPv + (b >> 1)], (uint32_t)((i - 1) & 1), abort_flag, p.status)) {
          alive = false;
          break;
        }
        // blocks 4-7 of the first tile held the f32 q rows until they were converted
        if (i == 0 && b == 4 && !wait_phase(&bars[kBarQc], 0, abort_flag, p.status)) {
          alive = false;
          break;
        }
        const uint32_t dst0 = sbase + kTOffK + b * kTBlockBytes;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          const int row = rsub + 16 * s;
          const uint32_t dst = dst0 + sw128(row, ch);
          if (prow[s] >= 0) {
            cp_async_16_plain(dst, b == 8 ? esrc[s] : ksrc[s] + b * 64);
          } else {
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0u) : "memory");
          }
        }
        cp_async_commit();
        if (b >= kTLag) {
          cp_async_wait<kTLag>();
          fence_proxy_async_smem();
          mbar_arrive(&bars[kBarFull + b - kTLag]);
        }
      }
      if (!alive) break;
      if (i + 1 < n_tiles) lookup(i + 1, pnext);  // the next tile's page ids, while the last groups fly
      cp_async_wait<0>();
      fence_proxy_async_smem();
      for (int b = kTBlocks - kTLag; b < kTBlocks; ++b) mbar_arrive(&bars[kBarFull + b]);
    }
    cp_async_wait<0>();
  }
  if (warp == kTMmaWarp) {
    // ---------------------------------------------------------------------- MMA
    constexpr uint32_t fmt = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
    constexpr uint32_t id_qk = instr_desc(fmt, 128, 64, false);
    constexpr uint32_t id_pv = instr_desc(fmt, 128, 64, true);
    const uint32_t k_addr = sbase + kTOffK, q_addr = sbase + kTOffQ, p_addr = sbase + kTOffP;
    bool alive = q_ok && (n_tiles == 0 || wait_phase(&bars[kBarQc], 0, abort_flag, p.status));
    bool issued = false;
    for (int i = 0; i < n_tiles && alive; ++i) {
      const uint32_t par = (uint32_t)(i & 1);
      // S^T = K . [Q_hi ; Q_lo]^T, blocks in the order they are refilled
      for (int bi = 0; bi < kTBlocks; ++bi) {
        const int b = bi;
        if (!wait_phase(&bars[kBarFull + b], par, abort_flag, p.status)) {
          alive = false;
          break;
        }
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t da = smem_desc(k_addr + b * kTBlockBytes + kk * 32, 16, 1024);
            const uint64_t db = smem_desc(q_addr + b * kTQBlockBytes + kk * 32, 16, 1024);
            umma(tmem + kColS, da, db, id_qk, (bi | kk) != 0);
          }
          issued = true;
        }
        __syncwarp();
      }
      if (!alive) break;
      if (lane == 0) umma_commit(&bars[kBarS]);
      __syncwarp();
      if (!wait_phase(&bars[kBarP], par, abort_flag, p.status)) break;
      tc_fence_after();
      // O^T += V^T . [P_hi ; P_lo]^T, one commit per 128-dim m-tile (frees latent blocks 2j, 2j+1)
      if (lane == 0) {
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
#pragma unroll
          for (int kt = 0; kt < 8; ++kt) {
            const uint64_t da = smem_desc(k_addr + (2 * j) * kTBlockBytes + kt * 2048, kTBlockBytes, 1024);
            const uint64_t db = smem_desc(p_addr + (kt >> 2) * kTPBlockBytes + (kt & 3) * 32, 16, 1024);
            umma(tmem + kColO + 64 * j, da, db, id_pv, (i | kt) != 0);
          }
          umma_commit(&bars[kBarPv + j]);
        }
      }
      __syncwarp();
    }
    // every MMA of this CTA has completed before tensor memory is released
    if (lane == 0 && issued) umma_commit(&bars[kBarDrain]);
    __syncwarp();
    if (__shfl_sync(0xffffffffu, issued ? 1 : 0, 0)) {
      if (!mbar_wait_bounded(&bars[kBarDrain], 0, kWaitLimitCycles) && lane == 0)
        report(p.status, PA_DEVICE_WAIT_TIMEOUT);
    }
    __syncwarp();
  } else if (warp >= kTSoftWarp0) {
    // ------------------------------------------------------------------ softmax
    const int wq = warp - kTSoftWarp0;      // lane quarter of tensor memory
    const int row = wq * 32 + lane;         // tile row = tensor-memory lane
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    float l_part[kTHeads];
#pragma unroll
    for (int h = 0; h < kTHeads; ++h) l_part[h] = 0.f;
    float m_lane = -INFINITY;  // running maximum of head `lane`
    bool alive = q_ok;
    unsigned char* pt = smem + kTOffP + (row >> 6) * kTPBlockBytes;
    for (int i = 0; i < n_tiles; ++i) {
      const uint32_t par = (uint32_t)(i & 1);
      if (!wait_phase(&bars[kBarS], par, abort_flag, p.status)) {
        alive = false;
        break;
      }
      tc_fence_after();
      int slot, e;
      const bool valid = chunk_row(p, gm, i * kTRows + row, &slot, &e);
      // per-head maximum over the tile's 128 rows (S^T is read again for P below,
      // which keeps the register peak low)
      float mt;
      {
        uint32_t hi[32], lo[32];
        __syncwarp();
        tmem_ld32(t_lane + kColS, hi);
        tmem_ld32(t_lane + kColS + 32, lo);
        float v[kTHeads];
#pragma unroll
        for (int h = 0; h < kTHeads; ++h)
          v[h] = valid ? __uint_as_float(hi[h]) + __uint_as_float(lo[h]) : -INFINITY;
        mt = reduce_scatter32<true>(v, lane);
      }
      red[(par * 4 + wq) * kTHeads + lane] = mt;
      mbar_arrive(&bars[kBarRed]);
      if (!wait_phase(&bars[kBarRed], par, abort_flag, p.status)) {
        alive = false;
        break;
      }
#pragma unroll
      for (int w = 0; w < 4; ++w) mt = fmaxf(mt, red[(par * 4 + w) * kTHeads + lane]);
      const bool need = mt > m_lane + kTLazy;
      const float m_new = need ? mt : m_lane;
      const float a_lane = need ? (m_lane == -INFINITY ? 0.f : fast_exp2(m_lane - m_new)) : 1.f;
      m_lane = m_new;
      const float mu_lane = m_lane == -INFINITY ? 0.f : m_lane;
      if (i > 0 && __any_sync(0xffffffffu, need)) {
        // raise the offsets: rescale O^T (all four m-tiles) and the row sums
        float a[kTHeads];
#pragma unroll
        for (int h = 0; h < kTHeads; ++h) a[h] = __shfl_sync(0xffffffffu, a_lane, h);
#pragma unroll 1
        for (int col = 0; col < 8; ++col) {  // m-tile col / 2, hi (even) or lo (odd) half
          uint32_t o[32];
          __syncwarp();
          tmem_ld32(t_lane + kColO + 32 * col, o);
#pragma unroll
          for (int h = 0; h < kTHeads; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * a[h]);
          tmem_st32(t_lane + kColO + 32 * col, o);
        }
#pragma unroll
        for (int h = 0; h < kTHeads; ++h) l_part[h] *= a[h];
      }
      // P = exp2(s - offset) in the pool's 16-bit type, written as P^T [head][token]
      uint32_t hi[32], lo[32];
      __syncwarp();
      tmem_ld32(t_lane + kColS, hi);
      tmem_ld32(t_lane + kColS + 32, lo);
#pragma unroll
      for (int h = 0; h < kTHeads; ++h) {
        const float mu = __shfl_sync(0xffffffffu, mu_lane, h);
        const float sc = valid ? __uint_as_float(hi[h]) + __uint_as_float(lo[h]) : -INFINITY;
        const float pr = fast_exp2(sc - mu);
        const float phi = TC<T>::round(pr);
        l_part[h] += pr;
        const uint32_t off = sw128(h, (row & 63) >> 3) + (row & 7) * 2;  // row h + 32: same swizzle phase
        *reinterpret_cast<unsigned short*>(pt + off) = TC<T>::bits(phi);
        *reinterpret_cast<unsigned short*>(pt + kTHeads * 128 + off) = TC<T>::bits(pr - phi);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars[kBarP]);
    }

    // ---- epilogue: row sums -> per-head totals, O^T -> normalized output rows ----
    if (alive && n_tiles > 0) {
      if (!wait_phase(&bars[kBarPv + 3], (uint32_t)((n_tiles - 1) & 1), abort_flag, p.status)) alive = false;
    }
    float L = 0.f;
    if (alive) {
      const uint32_t par = (uint32_t)(n_tiles & 1);
      const float lw = reduce_scatter32<false>(l_part, lane);
      red[(par * 4 + wq) * kTHeads + lane] = lw;
      mbar_arrive(&bars[kBarRed]);
      if (wait_phase(&bars[kBarRed], par, abort_flag, p.status)) {
#pragma unroll
        for (int w = 0; w < 4; ++w) L += red[(par * 4 + w) * kTHeads + lane];
      } else {
        alive = false;
      }
    }
    if (alive) {
      tc_fence_after();
      const float mu_lane = m_lane == -INFINITY ? 0.f : m_lane;
      const float inv_lane = L > 0.f ? 1.f / L : 0.f;
      if (wq == 0 && lane < nheads)
        p.lse_out[(size_t)c * p.num_qo_heads + h_first + lane] = L > 0.f ? mu_lane + fast_log2(L) : -INFINITY;
      float inv[kTHeads];
#pragma unroll
      for (int h = 0; h < kTHeads; ++h) inv[h] = __shfl_sync(0xffffffffu, inv_lane, h);
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        uint32_t o[32], ol[32];
        if (n_tiles > 0) {
          __syncwarp();
          tmem_ld32(t_lane + kColO + 64 * j, o);
          tmem_ld32(t_lane + kColO + 64 * j + 32, ol);
        } else {
#pragma unroll
          for (int h = 0; h < kTHeads; ++h) o[h] = ol[h] = 0u;
        }
        float* dst = p.v_out + ((size_t)c * p.num_qo_heads + h_first) * kTDim + j * 128 + row;
#pragma unroll
        for (int h = 0; h < kTHeads; ++h)
          if (h < nheads) dst[(size_t)h * kTDim] = (__uint_as_float(o[h]) + __uint_as_float(ol[h])) * inv[h];
      }
    }
  }

  // ---- release tensor memory once every role is done with it ----
  tc_fence_before();
  __syncwarp();
  __syncthreads();
  if (warp == kTMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// Self-test of the waits above (no tensor memory, no copies): warp 0 waits on a
// barrier nothing arrives on with a short limit and gives up; warp 1 waits on
// another with the full limit and must give up through the abort flag warp 0
// set.  completed[w] = 1 if warp w's wait returned true (it must not).
__global__ void __launch_bounds__(64, 1) pa_selftest_wait_kernel(int32_t* status, int32_t* completed,
                                                                  long long short_limit) {
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ uint32_t abort_word;
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    abort_word = 0u;
    fence_barrier_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  volatile uint32_t* abort_flag = &abort_word;
  const bool ok = warp == 0 ? wait_phase(&bars[0], 0, abort_flag, status, short_limit)
                            : wait_phase(&bars[1], 0, abort_flag, status, kWaitLimitCycles);
  if ((threadIdx.x & 31) == 0) completed[warp] = ok ? 1 : 0;
}

using Tc05Kernel = void (*)(const PartialParams, const Tc05Fields);

Tc05Kernel tc05_pick(int kv_dtype) {
  if (kv_dtype == PA_F16) return pa_v2_partial_extra_tc05_kernel<__half>;
  if (kv_dtype == PA_BF16) return pa_v2_partial_extra_tc05_kernel<__nv_bfloat16>;
  return nullptr;
}

}  // namespace

int occupancy_partial_extra_tc05(int kv_dtype, int* blocks_per_sm) {
  Tc05Kernel fn = tc05_pick(kv_dtype);
  if (!fn) return PA_EUNSUPPORTED;
  if (!prepare_kernel(reinterpret_cast<const void*>(fn), kTSmemAlloc)) return PA_ECUDA;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, fn, kTThreads, kTSmemAlloc) == cudaSuccess
             ? PA_OK
             : PA_ECUDA;
}

int launch_partial_extra_tc05(const PartialParams& p, const void* q_extra, const void* k_extra, int64_t k_stride,
                              int64_t e_stride, int kv_dtype, dim3 grid, cudaStream_t stream) {
  Tc05Kernel fn = tc05_pick(kv_dtype);
  if (!fn || p.hpc > kTHeads) return PA_EUNSUPPORTED;
  if (!prepare_kernel(reinterpret_cast<const void*>(fn), kTSmemAlloc)) return PA_ECUDA;
  Tc05Fields x;
  x.q_extra = static_cast<const float*>(q_extra);
  x.k_extra = k_extra;
  x.k_stride = k_stride;
  x.e_stride = e_stride;
  const cudaError_t rc = launch_dependent(fn, grid, dim3(kTThreads), kTSmemAlloc, stream, p, x);
  return rc == cudaSuccess && cudaGetLastError() == cudaSuccess ? PA_OK : PA_ECUDA;
}

}  // namespace pa

extern "C" pa_status pa_v2_selftest_wait(int32_t* status, int32_t* completed, int64_t limit_cycles,
                                         void* cuda_stream) {
  if (!status || !completed || limit_cycles < 1024 || limit_cycles > pa::kWaitLimitCycles) return PA_EINVAL;
  pa::pa_selftest_wait_kernel<<<1, 64, 0, static_cast<cudaStream_t>(cuda_stream)>>>(status, completed,
                                                                                    (long long)limit_cycles);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ECUDA;
}
