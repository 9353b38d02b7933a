// gemm_select.cu -- batched queries: bf16 tensor-core scoring with the top-K
// selection fused into the epilogue.
//
// For a batch of queries the scoring S = Q * C^T is a dense contraction, so it
// runs on the 5th-generation tensor cores (tcgen05): bf16 inputs, fp32
// accumulators in tensor memory (TMEM). The selection is the same problem as
// the single-query path (GPU-Resident Top-K for Agentic RAG, section 4 steps
// 3-4: per-block partial top-K, then a merge): every CTA pair leaves one
// best-first list per query, and the merge kernel finishes each query.
//
// One kernel, gemm_select_pair_kernel: clusters of two CTAs, one CTA per
// SM, 10 warps each, tcgen05.mma.cta_group::2 with M = 256 queries (128 per
// CTA) and N = 256 corpus rows (128 per CTA), 6 stages of 32 KB; it serves
// every batch size and K and the bound pre-pass.
// Per CTA:
//   warp 0     TMA producer: per 128-byte K chunk (64 bf16 or 32 fp32
//              elements) the CTA's queries and corpus rows, 128-byte
//              swizzled, into the shared-memory ring. The bf16 corpus is
//              stored tile-major ([row tile][K chunk][128 rows][64]), so each
//              corpus load is one contiguous 16 KB block of HBM;
//   warp 1     TMEM owner (both CTAs allocate as a pair); in the even CTA
//              one thread issues the pair's MMAs into one of two
//              accumulator buffers, so the epilogue drains tile t while
//              tile t + 1 accumulates;
//   warps 2-9  epilogue: thread = one query (its TMEM lane) over 128 of the
//              tile's columns; it marks the scores that may beat its K-th
//              best, buffers their keys 16 deep in shared memory and merges
//              full buffers into its best-first list: KP <= 32 keys in
//              registers, or for K > 32 a list in global memory (the
//              thread's slot of the partials buffer) with its length. At
//              the end the two warps on the same lanes merge their K <= 32
//              lists, so a query gets one list per CTA pair.
// The scores never reach memory: each thread writes one list per query. In
// bound mode (the pre-pass over a row sample) it writes instead the best key
// of each of its four 32-column chunks, folded over its tiles.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "rbf_device.cuh"
#include "rbf_internal.h"

namespace rbf {
namespace {

constexpr int kTileRows = 128;      // corpus rows per tile (MMA N)
constexpr int kKChunk = 64;         // bf16 elements per 128-byte swizzle row
constexpr int kKChunkTf32 = 32;     // fp32 (tf32) elements per 128-byte swizzle row
constexpr int kMmaPerChunk = 4;     // MMAs per 128-byte row: K = 16 bf16 or 8 tf32, 32 bytes each
constexpr int kSubTileBytes = 128 * kKChunk * 2;  // 16 KB: 128 rows x 128 B
constexpr int kCandCap = 16;        // buffered candidates per query
constexpr int kEpiWarps = 8;
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr int kTmemCols = 512;      // 2 buffers x 2 M tiles x 128 columns

// ------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 64 consecutive fp32 columns of this thread's TMEM lane, waited for.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes, groups of 8 rows 1024 bytes
// apart (stride byte offset), leading byte offset unused (1), descriptor
// version 1, layout SWIZZLE_128B (2). The tile base is 1024-byte aligned.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(const void* tile) {
  const uint32_t a = smem_addr(tile);
  uint64_t d = static_cast<uint64_t>((a >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor: fp32 accumulator (bits 4-5 = 1), the A and B
// formats (bits 7-9 and 10-12: 1 = bf16 for kind::f16, 2 = tf32 for
// kind::tf32), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n, uint32_t fmt) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// Elements of one 64 x 128-byte K chunk and the operand format code.
template <bool TF32>
struct Operand {
  static constexpr int kChunk = TF32 ? kKChunkTf32 : kKChunk;
  static constexpr uint32_t kFmt = TF32 ? 2u : 1u;
};

// ------------------------------------------------- per-thread key lists

// Descending bitonic sort of N (a power of two) keys in registers.
template <int N>
__device__ __forceinline__ void sort_desc(uint64_t (&c)[N]) {
#pragma unroll
  for (int k = 2; k <= N; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
      for (int i = 0; i < N; ++i) {
        const int l = i ^ j;
        if (l > i) {
          const uint64_t a = c[i], b = c[l];
          const bool desc = (i & k) == 0;
          c[i] = desc ? umax64(a, b) : umin64(a, b);
          c[l] = desc ? umin64(a, b) : umax64(a, b);
        }
      }
    }
  }
}

// Fold 8 sorted candidates onto the last 8 slots of a descending list of KP
// keys (reversed max) and restore the order with a bitonic merge.
template <int KP>
__device__ __forceinline__ void list_merge8(uint64_t (&L)[KP], const uint64_t (&c)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) L[KP - 8 + i] = umax64(L[KP - 8 + i], c[7 - i]);
#pragma unroll
  for (int j = KP / 2; j > 0; j >>= 1) {
#pragma unroll
    for (int i = 0; i < KP; ++i) {
      if ((i & j) == 0) {
        const uint64_t a = L[i], b = L[i + j];
        L[i] = umax64(a, b);
        L[i + j] = umin64(a, b);
      }
    }
  }
}

// Sort a bitonic sequence of KP keys in registers into descending order.
template <int KP>
__device__ __forceinline__ void bitonic_clean_desc(uint64_t (&L)[KP]) {
#pragma unroll
  for (int j = KP / 2; j > 0; j >>= 1) {
#pragma unroll
    for (int i = 0; i < KP; ++i) {
      if ((i & j) == 0) {
        const uint64_t a = L[i], b = L[i + j];
        L[i] = umax64(a, b);
        L[i + j] = umin64(a, b);
      }
    }
  }
}

template <int KP>
__device__ __forceinline__ uint64_t list_get(const uint64_t (&L)[KP], int e) {
  uint64_t x = 0;
#pragma unroll
  for (int i = 0; i < KP; ++i)
    if (i == e) x = L[i];
  return x;
}

// Write the warp's 32 lists of 32 keys (lane i's list is key_at(0..31) of
// lane i, to dst of lane i; no write for a null dst) with one 256-byte store
// of the warp per list instead of 32 scattered ones: the rows go through tr,
// 32 x 33 keys of shared memory that nothing else uses now.
template <typename KeyAt>
__device__ __forceinline__ void store_lists32(uint64_t* tr, int lane, uint64_t* dst, KeyAt key_at) {
#pragma unroll
  for (int i = 0; i < 32; ++i) tr[lane * 33 + i] = key_at(i);
  __syncwarp();
#pragma unroll 4
  for (int j = 0; j < 32; ++j) {
    uint64_t* d = reinterpret_cast<uint64_t*>(
        __shfl_sync(kFullMask, static_cast<unsigned long long>(reinterpret_cast<uintptr_t>(dst)), j));
    if (d) d[lane] = tr[j * 33 + lane];
  }
  __syncwarp();
}

// sc[j] for a warp-uniform j: a switch keeps the scores in registers (a
// dynamically indexed register array would live in local memory).
__device__ __forceinline__ float pick(const float (&sc)[32], int j) {
  switch (j) {
#define RBF_PICK(i) \
  case i:           \
    return sc[i];
    RBF_PICK(0) RBF_PICK(1) RBF_PICK(2) RBF_PICK(3) RBF_PICK(4) RBF_PICK(5) RBF_PICK(6) RBF_PICK(7)
    RBF_PICK(8) RBF_PICK(9) RBF_PICK(10) RBF_PICK(11) RBF_PICK(12) RBF_PICK(13) RBF_PICK(14) RBF_PICK(15)
    RBF_PICK(16) RBF_PICK(17) RBF_PICK(18) RBF_PICK(19) RBF_PICK(20) RBF_PICK(21) RBF_PICK(22) RBF_PICK(23)
    RBF_PICK(24) RBF_PICK(25) RBF_PICK(26) RBF_PICK(27) RBF_PICK(28) RBF_PICK(29) RBF_PICK(30)
#undef RBF_PICK
    default:
      return sc[31];
  }
}

struct Params {
  uint64_t* partials;  // [queries][grid / 2][32] keys; K > 32: [queries][grid][KP], lens[queries][grid] long;
                       // bound mode: [queries][grid][4]
  int* err;
  int64_t n;           // corpus rows
  int kchunks;         // 128-byte K chunks per row (64 bf16 or 32 fp32 elements)
  int q_row0;          // first query row of this launch in the bf16 query buffer
  int q_count;         // queries in this launch
  int q_out0;          // first query of this launch in the partials layout
  int k;
  uint64_t timeout_ns;
  const uint64_t* theta0;  // optional per-query lower bound on the K-th key
  int bound_mode;          // 1 (CTA pairs, KP = 8): write 4 chunk maxima per list instead of a top-K list
  int* lens;               // K > 32: valid keys of each list
  int wait_inputs;         // 1: the queries come from the kernel launched just before this one
  size_t partials_cap;     // keys, lens entries and theta0 entries, for checked builds
  size_t lens_cap;         // (0: not checked)
  size_t theta_cap;
  uint32_t index_offset;   // added to every row index (global rows of a shard)
};

// ------------------------------------------------ CTA pairs (2 SMs)
//
// A cluster of two CTAs computes each 256-row corpus tile against up to 256
// queries with tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16). Per
// 128-byte K chunk each CTA stages only its own 128 queries (A) and 128 of
// the tile's rows (B), 32 KB, so six stages fit; the MMA reads both CTAs'
// shared memory and writes each CTA's TMEM (its 128 queries x 256 rows). The
// even CTA of the pair issues the MMAs and multicasts each commit to both
// CTAs' barriers; the odd CTA's loads complete on the even CTA's full
// barrier, and both CTAs' epilogues release an accumulator on the even CTA's
// barrier. Lanes past the batch (up to 128 queries: the odd CTA's, and the
// padding of a partial group) mark nothing. (A single-CTA variant with two
// M tiles per CTA moved 1.5x the bytes per SM and stage for the same tensor
// work and could not cover a stage's round trip with four 48 KB stages.)

constexpr int kPairStages = 6;
constexpr int kPairStageBytes = 2 * kSubTileBytes;  // A (own 128 queries) | B (own 128 rows)
constexpr int kPairTileRows = 256;
constexpr int kPairAccArrivals = 2 * kEpiWarps;     // epilogue warps of both CTAs
// At the end the idle ring holds the epilogue warps' list transposes and the
// column-half list exchange.
static_assert(kPairStages * kPairStageBytes >= (kEpiWarps * 32 * 33 + 4 * 32 * 32) * 8, "ring too small");

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Shared::cluster address of the variable at `p` in the CTA of the given rank.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(p)), "r"(rank));
  return a;
}
// Arrival on a barrier of either CTA of the cluster that orders no memory:
// it only says that the arriving warp's TMEM loads have completed
// (tcgen05.wait::ld returned and tcgen05.fence::before_thread_sync issued),
// and a release at cluster scope would cost a fence per arrival.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
template <bool TF32>
__device__ __forceinline__ void umma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  if constexpr (TF32) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}
// Arrive once on `bar` in both CTAs of the pair when every MMA issued so far
// is done.
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_addr(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}
// Tiled TMA loads into this CTA's shared memory whose completion is counted
// on the barrier at cluster address `bar` (the even CTA's).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(map), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

template <int KP, bool TF32>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_select_pair_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_c,
                            const Params p) {
  constexpr int CH = Operand<TF32>::kChunk;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint64_t* cand = reinterpret_cast<uint64_t*>(smem + kPairStages * kPairStageBytes);  // [kCandCap][256]
  uint64_t* full = cand + kCandCap * 256;
  uint64_t* empty = full + kPairStages;
  uint64_t* acc_full = empty + kPairStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = static_cast<int>(blockIdx.x >> 1);
  const int nclusters = static_cast<int>(gridDim.x >> 1);
  const int num_pair_tiles = static_cast<int>((p.n + kPairTileRows - 1) / kPairTileRows);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&full[s], 1);   // the even CTA's producer (expect_tx for both CTAs' bytes)
      mbar_init(&empty[s], 1);  // one multicast commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kPairAccArrivals);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  // Both CTAs' barriers are initialised before either CTA signals the other.
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Launched as a programmatic dependent: the next kernel may be scheduled
  // now (it waits for this grid before it reads anything written here). The
  // corpus stream starts while the previous kernel finishes unless that
  // kernel wrote the queries; the epilogue waits for it before it reads the
  // bounds or writes any list.
  pdl_launch_dependents();

  if (warp == 0) {
    // --------------------------------------------------------- TMA producer
    if (lane == 0) {
      if (p.wait_inputs) pdl_wait();
      const uint64_t pol_c = l2_policy_evict_first();
      const uint64_t pol_q = l2_policy_evict_last();
      int64_t it = 0;
      bool aborted = false;
      for (int t = cluster; t < num_pair_tiles && !aborted; t += nclusters) {
        for (int kc = 0; kc < p.kchunks; ++kc, ++it) {
          const int s = static_cast<int>(it % kPairStages);
          const uint32_t u = static_cast<uint32_t>(it / kPairStages);
          if (u > 0 && !mbar_wait(&empty[s], (u - 1) & 1u, p.timeout_ns)) {
            atomicOr(p.err, kErrProducerTimeout);
            aborted = true;
            break;
          }
          if (*reinterpret_cast<volatile int*>(&abort_flag)) {
            aborted = true;
            break;
          }
          uint8_t* st = ring + static_cast<size_t>(s) * kPairStageBytes;
          if (leader) mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(2 * kPairStageBytes));
          const uint32_t bar = cluster_addr(&full[s], 0);
          tma_load_2d_pair(st, &tmap_q, kc * CH, p.q_row0 + static_cast<int>(rank) * 128, bar, pol_q);
          if constexpr (TF32)
            tma_load_2d_pair(st + kSubTileBytes, &tmap_c, kc * CH, (2 * t + static_cast<int>(rank)) * kTileRows, bar,
                             pol_c);
          else
            tma_load_3d_pair(st + kSubTileBytes, &tmap_c, 0, 0, (2 * t + static_cast<int>(rank)) * p.kchunks + kc, bar,
                             pol_c);
        }
      }
      if (aborted) {
        abort_flag = 1;
        // The even CTA lets every stage it armed land before the pair can exit
        // (those phases count both CTAs' loads).
        if (leader) {
          for (int64_t i = (it > kPairStages ? it - kPairStages : 0); i < it; ++i) {
            const int s = static_cast<int>(i % kPairStages);
            if (!mbar_wait(&full[s], static_cast<uint32_t>(i / kPairStages) & 1u, p.timeout_ns))
              atomicOr(p.err, kErrDrainTimeout);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      if (leader) {
        constexpr uint32_t idesc = make_idesc(256, kPairTileRows, Operand<TF32>::kFmt);
        int64_t it = 0;
        int tile_i = 0;
        bool aborted = false;
        for (int t = cluster; t < num_pair_tiles && !aborted; t += nclusters, ++tile_i) {
          const int b = tile_i & 1;
          const uint32_t ub = static_cast<uint32_t>(tile_i >> 1);
          if (ub > 0 && !mbar_wait(&acc_empty[b], (ub - 1) & 1u, p.timeout_ns)) {
            atomicOr(p.err, kErrConsumerTimeout);
            aborted = true;
            break;
          }
          tc_fence_after();
          for (int kc = 0; kc < p.kchunks; ++kc, ++it) {
            const int s = static_cast<int>(it % kPairStages);
            if (!mbar_wait(&full[s], static_cast<uint32_t>(it / kPairStages) & 1u, p.timeout_ns)) {
              atomicOr(p.err, kErrConsumerTimeout);
              aborted = true;
              break;
            }
            tc_fence_after();
            const uint8_t* st = ring + static_cast<size_t>(s) * kPairStageBytes;
            const uint64_t adesc = sw128_kmajor_desc(st);
            const uint64_t bdesc = sw128_kmajor_desc(st + kSubTileBytes);
            const uint32_t d = tmem_base + static_cast<uint32_t>(b * kPairTileRows);
#pragma unroll
            for (int k = 0; k < kMmaPerChunk; ++k)
              umma_pair<TF32>(d, adesc + static_cast<uint64_t>(2 * k), bdesc + static_cast<uint64_t>(2 * k), idesc,
                              (kc | k) != 0);
            umma_commit_pair(&empty[s]);  // both CTAs' stage s is free once these MMAs finish
          }
          if (aborted) break;
          umma_commit_pair(&acc_full[b]);  // both CTAs' accumulators are complete
        }
        if (aborted) abort_flag = 1;
        // Every MMA (they read both CTAs' shared memory and write both TMEMs)
        // must be finished before either CTA releases TMEM or exits.
        umma_commit_pair(drain);
      }
      if (!mbar_wait(drain, 0, p.timeout_ns)) atomicOr(p.err, kErrDrainTimeout);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- epilogue
    pdl_wait();
    const int e = warp - 2;
    const int quad = warp & 3;        // TMEM lane quadrant this warp may access
    const int h = e >> 2;             // which 128 of the tile's 256 rows
    const int qlocal = quad * 32 + lane;
    const int qidx = static_cast<int>(rank) * 128 + qlocal;  // query within this launch
    const int slot = h * 128 + qlocal;                        // candidate buffer column
    const uint32_t acc_empty_leader0 = cluster_addr(&acc_empty[0], 0);
    const uint32_t acc_empty_leader1 = cluster_addr(&acc_empty[1], 0);
    // K <= 32: the thread's best-first list of KP keys is in registers.
    // K > 32 (KP = 64, 128 or 256): it is the thread's own partials list in
    // global memory, `len` keys long, and buffered candidates are merged into
    // it from the back; on random data with the sample bound only a few dozen
    // keys per thread ever reach it.
    constexpr bool kWide = KP > 32;
    uint64_t L[kWide ? 1 : KP];
#pragma unroll
    for (int i = 0; i < (kWide ? 1 : KP); ++i) L[i] = 0;
    auto list_id = [&]() {
      return static_cast<size_t>(p.q_out0 + qidx) * gridDim.x + static_cast<size_t>(cluster * 2 + h);
    };
    // A lane past the batch, or (checked builds) one whose list would fall
    // outside the buffers, marks nothing and writes nothing.
    const bool live =
        qidx < p.q_count &&
        in_bounds(p.partials_cap == 0 || (list_id() + 1) * (kWide ? KP : 32) <= p.partials_cap, p.err) &&
        in_bounds(!kWide || p.lens_cap == 0 || list_id() < p.lens_cap, p.err) &&
        in_bounds(!p.theta0 || p.theta_cap == 0 || static_cast<size_t>(p.q_row0 + qidx) < p.theta_cap, p.err);
    uint64_t* lst = nullptr;
    if constexpr (kWide) lst = p.partials + list_id() * KP;
    int len = 0;
    uint64_t floor_key = 0;
    if (p.theta0 && live) {
      const uint64_t b0 = p.theta0[p.q_row0 + qidx];
      floor_key = b0 > 0 ? b0 - 1 : 0;
    }
    uint64_t theta = floor_key;
    float theta_f = floor_key ? key_score(floor_key + 1) : 0.0f;
    bool filling = floor_key == 0;
    int cnt = 0;
    // Bound mode (KP = 8 instance only): the best key of each of the 4
    // 32-row chunks of the thread's 128 columns, folded over its tiles.
    uint64_t best[4] = {0ull, 0ull, 0ull, 0ull};
    const bool bound = KP == 8 && p.bound_mode;

    auto merge_buffer = [&]() {
      if constexpr (kWide) {
        if (cnt > 0) {
          uint64_t c[kCandCap];
#pragma unroll
          for (int i = 0; i < kCandCap; ++i) c[i] = i < cnt ? cand[i * 256 + slot] : 0ull;
          sort_desc(c);
          // Merge into the list without a chain of dependent loads: list
          // key x moves up by s(x) = the number of candidates above it, and
          // candidate j lands at j + the number of list keys above it.
          // Keys are read back to front, kScan independent loads at a time,
          // and moved (at most K kept); the scan stops at the first batch
          // that reaches a key no candidate beats (it and everything before
          // it stay). above[j / 2] counts, in its low or high 16 bits, the
          // scanned keys above candidate j.
          constexpr int kScan = 4;
          uint32_t above[kCandCap / 2];
#pragma unroll
          for (int j = 0; j < kCandCap / 2; ++j) above[j] = 0;
          int i = len;
#pragma unroll 1
          while (i > 0) {
            const int i0 = i > kScan ? i - kScan : 0;
            uint64_t x[kScan];
#pragma unroll
            for (int u = 0; u < kScan; ++u) x[u] = i0 + u < i ? lst[i0 + u] : ~0ull;
            bool reached = false;
#pragma unroll
            for (int u = kScan - 1; u >= 0; --u) {
              int sh = 0;
#pragma unroll
              for (int j = 0; j < kCandCap; ++j) sh += c[j] > x[u] ? 1 : 0;
              const bool valid = i0 + u < i;
              reached |= valid && sh == 0;
              if (valid && sh > 0 && i0 + u + sh < p.k) lst[i0 + u + sh] = x[u];
#pragma unroll
              for (int j = 0; j < kCandCap; ++j)
                above[j / 2] += (valid && sh <= j) ? (1u << (16 * (j & 1))) : 0u;
            }
            i = i0;
            if (reached) break;
          }
#pragma unroll
          for (int j = 0; j < kCandCap; ++j) {
            const int at = j + i + static_cast<int>((above[j / 2] >> (16 * (j & 1))) & 0xFFFFu);
            if (j < cnt && at < p.k) lst[at] = c[j];
          }
          len = min(len + cnt, p.k);
          cnt = 0;
          if (len == p.k) {
            theta = umax64(lst[p.k - 1], floor_key);
            filling = theta == 0;
            theta_f = filling ? 0.0f : key_score(theta == floor_key ? floor_key + 1 : theta);
          }
        }
      } else {
        const int batches = static_cast<int>((__reduce_max_sync(kFullMask, static_cast<unsigned>(cnt)) + 7u) >> 3);
#pragma unroll 1
        for (int b8 = 0; b8 < batches * 8; b8 += 8) {
          uint64_t c[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) c[i] = (b8 + i < cnt) ? cand[(b8 + i) * 256 + slot] : 0ull;
          sort_desc(c);
          list_merge8<KP>(L, c);
        }
        cnt = 0;
        theta = umax64(list_get<KP>(L, p.k - 1), floor_key);
        filling = theta == 0;
        theta_f = filling ? 0.0f : key_score(theta == floor_key ? floor_key + 1 : theta);
      }
    };

    int tile_i = 0;
    for (int t = cluster; t < num_pair_tiles; t += nclusters, ++tile_i) {
      const int b = tile_i & 1;
      if (!__all_sync(kFullMask, mbar_wait(&acc_full[b], static_cast<uint32_t>(tile_i >> 1) & 1u, p.timeout_ns))) {
        if (lane == 0) atomicOr(p.err, kErrConsumerTimeout);
        abort_flag = 1;
        break;
      }
      if (__any_sync(kFullMask, *reinterpret_cast<volatile int*>(&abort_flag) != 0)) break;
      tc_fence_after();
      const int64_t row0 = static_cast<int64_t>(t) * kPairTileRows + h * 128;
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             static_cast<uint32_t>(b * kPairTileRows + h * 128);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float s64[64];
        tmem_ld64(tbase + static_cast<uint32_t>(hh * 64), s64);
        if (hh == 1) {
          // The accumulator may be overwritten from here on: release it on
          // the even CTA's barrier.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(b ? acc_empty_leader1 : acc_empty_leader0);
        }
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          const float(&sc)[32] = *reinterpret_cast<const float(*)[32]>(&s64[c2 * 32]);
          const int64_t rb = row0 + hh * 64 + c2 * 32;
          if constexpr (KP == 8) {
            if (bound) {
              // The chunk's best key: its largest score (NaN ignored) at the
              // first column holding it, one key built per chunk. Any row's
              // key of the chunk would keep the bound valid (K chunks give K
              // distinct rows); all-NaN chunks take their first row.
              const int64_t left = p.n - rb;
              const int nvalid = left >= 32 ? 32 : (left > 0 ? static_cast<int>(left) : 0);
              if (nvalid > 0) {
                float t16[16];
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  t16[j] = fmaxf(j < nvalid ? sc[j] : -INFINITY, j + 16 < nvalid ? sc[j + 16] : -INFINITY);
#pragma unroll
                for (int w = 8; w > 0; w >>= 1)
#pragma unroll
                  for (int j = 0; j < w; ++j) t16[j] = fmaxf(t16[j], t16[j + w]);
                const float mx = t16[0];
                uint32_t eq = 0;
#pragma unroll
                for (int j = 0; j < 32; ++j) eq |= (j < nvalid && sc[j] == mx) ? (1u << j) : 0u;
                const int jm = eq ? __ffs(eq) - 1 : 0;
                best[hh * 2 + c2] =
                    umax64(best[hh * 2 + c2], make_key(mx, static_cast<uint32_t>(rb + jm) + p.index_offset));
              }
              continue;
            }
          }
          uint32_t m = 0;
#pragma unroll
          for (int j = 0; j < 32; ++j) m |= (sc[j] >= theta_f) ? (1u << j) : 0u;
          if (filling) m = 0xFFFFFFFFu;
          if (p.n - rb < 32) m &= (p.n - rb > 0) ? ((1u << (p.n - rb)) - 1u) : 0u;
          if (!live) m = 0;
          uint32_t u = __reduce_or_sync(kFullMask, m);
          while (u) {
            const int j = __ffs(u) - 1;
            u &= u - 1;
            if (m & (1u << j)) {
              const uint64_t key = make_key(pick(sc, j), static_cast<uint32_t>(rb + j) + p.index_offset);
              if (key > theta) {
                cand[cnt * 256 + slot] = key;
                ++cnt;
              }
            }
            if (__any_sync(kFullMask, cnt == kCandCap)) merge_buffer();
          }
        }
      }
    }
    if (bound) {
      // Best first (a 4-key sorting network), then zeros to the list width.
      auto cswap = [](uint64_t& x, uint64_t& y) {
        const uint64_t hi = umax64(x, y), lo = umin64(x, y);
        x = hi;
        y = lo;
      };
      cswap(best[0], best[1]);
      cswap(best[2], best[3]);
      cswap(best[0], best[2]);
      cswap(best[1], best[3]);
      cswap(best[1], best[2]);
      // Lists of kBoundListWidth (4) keys: two 16-byte stores per thread.
      if (live) {
        ulonglong2* dst = reinterpret_cast<ulonglong2*>(p.partials + list_id() * kBoundListWidth);
        dst[0] = make_ulonglong2(best[0], best[1]);
        dst[1] = make_ulonglong2(best[2], best[3]);
      }
    } else {
      if (__any_sync(kFullMask, cnt > 0)) merge_buffer();
      if constexpr (kWide) {
        if (live) p.lens[list_id()] = len;
      } else {
        // The two warps on the same TMEM lanes (column halves h = 0 and 1)
        // hold two lists per query. The h = 1 warp hands its list over
        // through shared memory (every MMA has finished, so the ring is
        // idle), and the h = 0 warp folds it into its own (reversed max, then
        // a bitonic merge) and writes one list per query and CTA pair.
        uint64_t* xch = reinterpret_cast<uint64_t*>(ring) + kEpiWarps * (32 * 33) + quad * (32 * KP);
        if (h == 1) {
#pragma unroll
          for (int i = 0; i < KP; ++i) xch[i * 32 + lane] = L[i];
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory");
        if (h == 0) {
#pragma unroll
          for (int i = 0; i < KP; ++i) L[KP - 1 - i] = umax64(L[KP - 1 - i], xch[i * 32 + lane]);
          bitonic_clean_desc<KP>(L);
          const size_t pair_list = static_cast<size_t>(p.q_out0 + qidx) * nclusters + cluster;
          store_lists32(reinterpret_cast<uint64_t*>(ring) + e * (32 * 33), lane,
                        live ? p.partials + pair_list * 32 : nullptr, [&](int i) { return i < KP ? L[i] : 0ull; });
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // Neither CTA releases TMEM or exits while the other may still signal it.
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

// --------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return nullptr;
  }();
  return fn;
}

int pair_smem_bytes() {
  return 1024 + kPairStages * kPairStageBytes + kCandCap * 256 * 8 + (2 * kPairStages + 5) * 8 + 16;
}

template <int KP, bool TF32>
cudaError_t launch_pair_t(const CUtensorMap& tq, const CUtensorMap& tc, const Params& p, int grid, cudaStream_t st) {
  auto fn = gemm_select_pair_kernel<KP, TF32>;
  const int smem = pair_smem_bytes();
  static PerDeviceOnce once;
  const cudaError_t limit =
      once.run([fn, smem] { return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); });
  if (limit != cudaSuccess) return limit;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, fn, tq, tc, p);
}

// fp32 [rows][src_pitch] -> bf16 [rows][dst_pitch], zero past `cols` and for
// rows in [rows, rows_total).
__global__ void to_bf16_kernel(const float* __restrict__ src, int64_t src_pitch, __nv_bfloat16* __restrict__ dst,
                               int64_t dst_pitch, int64_t rows, int64_t rows_total, int cols) {
  pdl_launch_dependents();  // the scoring pass may become resident now; its producer waits for these queries
  const int64_t total = rows_total * dst_pitch;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / dst_pitch;
    const int64_t c = i - r * dst_pitch;
    const float v = (r < rows && c < cols) ? src[r * src_pitch + c] : 0.0f;
    dst[i] = __float2bfloat16_rn(v);
  }
}

// As to_bf16_kernel, four elements per thread: one 16-byte load and one
// 8-byte store (src 16-byte aligned, src_pitch and dst_pitch multiples of 4);
// a row's last partial group of four is read element by element.
__global__ void to_bf16_x4_kernel(const float* __restrict__ src, int64_t src_pitch, __nv_bfloat16* __restrict__ dst,
                                  int64_t dst_pitch, int64_t rows, int64_t rows_total, int cols) {
  pdl_launch_dependents();  // the scoring pass may become resident now; its producer waits for these queries
  const int64_t total4 = rows_total * dst_pitch / 4;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = i * 4;
    const int64_t r = e / dst_pitch;
    const int c = static_cast<int>(e - r * dst_pitch);
    float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (r < rows) {
      const float* x = src + r * src_pitch + c;
      if (c + 3 < cols) {
        v = *reinterpret_cast<const float4*>(x);
      } else {
        if (c < cols) v.x = x[0];
        if (c + 1 < cols) v.y = x[1];
        if (c + 2 < cols) v.z = x[2];
      }
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 w;
    w.x = *reinterpret_cast<const uint32_t*>(&lo);
    w.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst + e) = w;
  }
}

// fp32 [rows][src_pitch] -> bf16 tile-major [tiles][kchunks][128][64], zero
// past `cols` and for rows in [rows, tiles * 128).
__global__ void to_bf16_tiled_kernel(const float* __restrict__ src, int64_t src_pitch,
                                     __nv_bfloat16* __restrict__ dst, int64_t rows, int64_t tiles, int kchunks,
                                     int cols) {
  const int64_t total = tiles * kchunks * (kTileRows * kKChunk);
  for (int64_t o = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; o < total;
       o += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int cc = static_cast<int>(o % kKChunk);
    const int rr = static_cast<int>((o / kKChunk) % kTileRows);
    const int64_t tk = o / (kTileRows * kKChunk);
    const int kc = static_cast<int>(tk % kchunks);
    const int64_t r = (tk / kchunks) * kTileRows + rr;
    const int c = kc * kKChunk + cc;
    const float v = (r < rows && c < cols) ? src[r * src_pitch + c] : 0.0f;
    dst[o] = __float2bfloat16_rn(v);
  }
}

}  // namespace

bool make_bf16_tensor_map(void* map_out, const void* base, int64_t rows, int pitch_elems) {
  CUtensorMap* map = static_cast<CUtensorMap*>(map_out);
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(pitch_elems), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch_elems) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kKChunk), 128};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_bf16_tiled_tensor_map(void* map_out, const void* base, int64_t rows, int pitch_elems) {
  CUtensorMap* map = static_cast<CUtensorMap*>(map_out);
  auto fn = encode_fn();
  if (!fn) return false;
  const int64_t blocks = (rows + kTileRows - 1) / kTileRows * (pitch_elems / kKChunk);
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kKChunk), static_cast<cuuint64_t>(kTileRows),
                              static_cast<cuuint64_t>(blocks)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kKChunk) * 2, static_cast<cuuint64_t>(kSubTileBytes)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kKChunk), static_cast<cuuint32_t>(kTileRows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_to_bf16_tiled(const float* src, int64_t src_pitch, void* dst, int64_t rows, int pitch_elems,
                                 int cols, int num_sms, cudaStream_t st) {
  const int64_t tiles = (rows + kTileRows - 1) / kTileRows;
  const int kchunks = pitch_elems / kKChunk;
  const int64_t total = tiles * kchunks * (kTileRows * kKChunk);
  int64_t blocks = (total + 255) / 256;
  blocks = blocks < int64_t(num_sms) * 8 ? blocks : int64_t(num_sms) * 8;
  if (blocks < 1) blocks = 1;
  to_bf16_tiled_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(src, src_pitch, static_cast<__nv_bfloat16*>(dst),
                                                                rows, tiles, kchunks, cols);
  return cudaGetLastError();
}

bool make_f32_tensor_map(void* map_out, const void* base, int64_t rows, int pitch_elems) {
  CUtensorMap* map = static_cast<CUtensorMap*>(map_out);
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(pitch_elems), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch_elems) * 4};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kKChunkTf32), 128};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_to_bf16(const float* src, int64_t src_pitch, void* dst, int64_t dst_pitch, int64_t rows,
                           int64_t rows_total, int cols, int num_sms, cudaStream_t st) {
  const bool x4 = (reinterpret_cast<uintptr_t>(src) & 15) == 0 && src_pitch % 4 == 0 && dst_pitch % 4 == 0 &&
                  (reinterpret_cast<uintptr_t>(dst) & 7) == 0;
  const int64_t total = rows_total * dst_pitch / (x4 ? 4 : 1);
  int64_t blocks = (total + 255) / 256;
  blocks = blocks < int64_t(num_sms) * 8 ? blocks : int64_t(num_sms) * 8;
  if (blocks < 1) blocks = 1;
  if (x4)
    to_bf16_x4_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(src, src_pitch, static_cast<__nv_bfloat16*>(dst),
                                                               dst_pitch, rows, rows_total, cols);
  else
    to_bf16_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(src, src_pitch, static_cast<__nv_bfloat16*>(dst),
                                                            dst_pitch, rows, rows_total, cols);
  return cudaGetLastError();
}

template <bool TF32>
cudaError_t launch_typed(const CUtensorMap& tq, const CUtensorMap& tc, const Params& p, const GemmSelectLaunch& a,
                         cudaStream_t stream) {
  if (a.grid < 2 || a.grid % 2 != 0) return cudaErrorInvalidValue;
  if (a.bound_mode) return launch_pair_t<8, TF32>(tq, tc, p, a.grid, stream);
  if (a.k > 32) {
    // Lists in global memory.
    if (!a.lens) return cudaErrorInvalidValue;
    // List stride list_width(K), as the merge reads it.
    if (a.k <= 64) return launch_pair_t<64, TF32>(tq, tc, p, a.grid, stream);
    if (a.k <= 128) return launch_pair_t<128, TF32>(tq, tc, p, a.grid, stream);
    if (a.k <= 256) return launch_pair_t<256, TF32>(tq, tc, p, a.grid, stream);
    return cudaErrorInvalidValue;
  }
  // Register lists (lists per query = grid), any number of queries up to 256.
  if (a.k <= 8) return launch_pair_t<8, TF32>(tq, tc, p, a.grid, stream);
  if (a.k <= 16) return launch_pair_t<16, TF32>(tq, tc, p, a.grid, stream);
  if (a.k <= 32) return launch_pair_t<32, TF32>(tq, tc, p, a.grid, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_select(const GemmSelectLaunch& a, cudaStream_t stream) {
  Params p;
  p.partials = a.partials;
  p.err = a.err;
  p.n = a.n;
  p.kchunks = a.kchunks;
  p.q_row0 = a.q_row0;
  p.q_count = a.q_count;
  p.q_out0 = a.q_out0;
  p.k = a.k;
  p.timeout_ns = a.timeout_ns;
  p.theta0 = a.theta0;
  p.bound_mode = a.bound_mode;
  p.lens = a.lens;
  p.wait_inputs = a.wait_inputs;
  p.partials_cap = a.partials_cap;
  p.lens_cap = a.lens_cap;
  p.theta_cap = a.theta_cap;
  p.index_offset = a.index_offset;
  const CUtensorMap& tq = *static_cast<const CUtensorMap*>(a.tmap_q);
  const CUtensorMap& tc = *static_cast<const CUtensorMap*>(a.tmap_c);
  return a.tf32 ? launch_typed<true>(tq, tc, p, a, stream) : launch_typed<false>(tq, tc, p, a, stream);
}

}  // namespace rbf
