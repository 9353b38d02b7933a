// topk_i32.cu -- stage 1 of the flat int32 two-stage top-K.
//
// CUDA programming model series 9 (sections 2.1-2.2): every block computes a
// local top-K over its share of the array, and stage 2 merges the GRID x K
// candidates in one block (the merge kernel here). That page keeps a sorted
// register array per thread and merges threads with a shared-memory tree;
// here each warp keeps one register bitonic list with a threshold instead:
//
//   * persistent grid; CTA b owns a contiguous range of 16-byte vectors;
//   * every lane issues four 16-byte streaming loads before using any of them
//     (2 KB in flight per warp), so the loop is bound by HBM, not latency;
//   * each value is keyed with its position; a key that beats the warp's K-th
//     best goes into a 64-entry shared-memory buffer via ballot compaction,
//     and every 32 buffered keys are merged into the list;
//   * the few elements before the first 16-byte boundary and after the last
//     one are handled by scalar loads in CTA 0;
//   * the CTA merges its warps' lists and writes one best-first list.
#include "merge_core.cuh"
#include "rbf_device.cuh"
#include "rbf_internal.h"

namespace rbf {
namespace {

constexpr int NW = kI32Warps;
constexpr int kUnroll = 4;

struct WarpBuffer {
  uint64_t slot[64];
};

// Append the keys that beat theta (one candidate per lane, `pass` per lane)
// to the warp buffer; merge 32 into the list whenever 32 or more are waiting.
template <int R>
__device__ __forceinline__ void offer(uint64_t (&v)[R], WarpBuffer& buf, int& cnt, uint64_t& theta, uint64_t floor_key,
                                      int k, uint64_t key, bool pass, int lane) {
  const unsigned mask = __ballot_sync(kFullMask, pass);
  if (mask == 0) return;
  const int rank = __popc(mask & ((1u << lane) - 1u));
  if (pass) buf.slot[cnt + rank] = key;
  cnt += __popc(mask);
  __syncwarp();
  if (cnt >= 32) {
    const uint64_t cand = buf.slot[lane];
    const uint64_t rest = buf.slot[32 + lane];
    __syncwarp();
    warp_list_insert32<R>(v, cand, lane);
    theta = umax64(warp_list_get<R>(v, k - 1), floor_key);
    cnt -= 32;
    if (lane < cnt) buf.slot[lane] = rest;
    __syncwarp();
  }
}

// One step of 4 x int4 per lane (16 values, positions pos_base + 4*32*q + 4*lane
// + j in the lane's view): a superset mask of the values that may beat theta
// (value code >= theta's, settled exactly by the key compare), a warp vote,
// and a walk over the union of flagged slots in which each lane offers the
// value in that slot if it flagged it. Slot b = 4*q + j.
template <int R>
__device__ __forceinline__ void scan16(uint64_t (&v)[R], WarpBuffer& buf, int& cnt, uint64_t& theta,
                                       uint64_t floor_key, int k, const int4 (&x)[4], const bool (&in)[4],
                                       const uint32_t (&pos)[4], int lane) {
  const uint32_t theta_hi = static_cast<uint32_t>(theta >> 32);
  uint32_t m = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (in[q]) {
      m |= ((static_cast<uint32_t>(x[q].x) ^ 0x80000000u) >= theta_hi ? 1u : 0u) << (4 * q + 0);
      m |= ((static_cast<uint32_t>(x[q].y) ^ 0x80000000u) >= theta_hi ? 1u : 0u) << (4 * q + 1);
      m |= ((static_cast<uint32_t>(x[q].z) ^ 0x80000000u) >= theta_hi ? 1u : 0u) << (4 * q + 2);
      m |= ((static_cast<uint32_t>(x[q].w) ^ 0x80000000u) >= theta_hi ? 1u : 0u) << (4 * q + 3);
    }
  }
  uint32_t u = __reduce_or_sync(kFullMask, m);
  while (u) {
    const int b = __ffs(u) - 1;
    u &= u - 1;
    const int q = b >> 2;
    int32_t val = 0;
    // A uniform switch picks the register (dynamic indexing would spill).
    switch (b) {
#define RBF_SLOT(i, f) \
  case i:              \
    val = x[i / 4].f;  \
    break;
      RBF_SLOT(0, x) RBF_SLOT(1, y) RBF_SLOT(2, z) RBF_SLOT(3, w) RBF_SLOT(4, x) RBF_SLOT(5, y) RBF_SLOT(6, z)
      RBF_SLOT(7, w) RBF_SLOT(8, x) RBF_SLOT(9, y) RBF_SLOT(10, z) RBF_SLOT(11, w) RBF_SLOT(12, x)
      RBF_SLOT(13, y) RBF_SLOT(14, z) RBF_SLOT(15, w)
#undef RBF_SLOT
    }
    uint32_t pq = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (i == q) pq = pos[i];
    const uint64_t key = make_ikey(val, pq + static_cast<uint32_t>(b & 3));
    offer<R>(v, buf, cnt, theta, floor_key, k, key, ((m >> b) & 1u) && key > theta, lane);
  }
}

template <int KP>
__global__ void __launch_bounds__(NW * 32) topk_i32_stage1_kernel(const int32_t* __restrict__ data, int64_t n,
                                                                  int k, uint64_t* partials,
                                                                  const uint64_t* __restrict__ theta0,
                                                                  size_t partials_cap, int* err) {
  constexpr int R = KP / 32;
  __shared__ WarpBuffer bufs[NW];
  __shared__ __align__(16) uint64_t lists[NW * KP];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  WarpBuffer& buf = bufs[warp];
  pdl_launch_dependents();

  // Split into scalar head | 16-byte vectors | scalar tail.
  const uintptr_t addr = reinterpret_cast<uintptr_t>(data);
  int64_t head = static_cast<int64_t>(((16 - (addr & 15)) & 15) >> 2);
  if (head > n) head = n;
  const int64_t nvec = (n - head) >> 2;
  const int64_t tail0 = head + nvec * 4;
  const int4* vec = reinterpret_cast<const int4*>(data + head);

  uint64_t v[R];
  warp_list_clear<R>(v);
  // theta: keys <= theta are dropped. With a lower bound b on the final K-th
  // key (the K-th best key of a sample of the array), keys >= b can still
  // make the top K, so theta starts at b - 1.
  uint64_t floor_key = 0;
  if (theta0) {
    const uint64_t b0 = *theta0;
    floor_key = b0 > 0 ? b0 - 1 : 0;
  }
  uint64_t theta = floor_key;
  int cnt = 0;

  const int64_t v0 = nvec * blockIdx.x / gridDim.x;
  const int64_t v1 = nvec * (blockIdx.x + 1) / gridDim.x;
  constexpr int64_t kChunk = 32 * kUnroll;  // vectors per warp step
  for (int64_t c = v0 + static_cast<int64_t>(warp) * kChunk; c < v1; c += static_cast<int64_t>(NW) * kChunk) {
    int4 x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = c + u * 32 + lane;
      x[u] = (i < v1) ? __ldcs(vec + i) : make_int4(0, 0, 0, 0);
    }
    bool in[kUnroll];
    uint32_t pos[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = c + u * 32 + lane;
      in[u] = i < v1;
      pos[u] = static_cast<uint32_t>(head + i * 4);
    }
    scan16<R>(v, buf, cnt, theta, floor_key, k, x, in, pos, lane);
  }
  if (blockIdx.x == 0 && warp == 0) {
    // Unaligned head and the tail: at most 3 + 3 elements.
    const int64_t extra = head + (n - tail0);
    for (int64_t b = 0; b < extra; b += 32) {
      const int64_t t = b + lane;
      bool in = t < extra;
      int64_t pos = 0;
      if (in) pos = (t < head) ? t : tail0 + (t - head);
      const uint64_t key = in ? make_ikey(data[pos], static_cast<uint32_t>(pos)) : 0;
      offer<R>(v, buf, cnt, theta, floor_key, k, key, in && key > theta, lane);
    }
  }
  // Flush what is left in the buffer (empty slots are the zero sentinel).
  if (cnt > 0) {
    const uint64_t cand = (lane < cnt) ? buf.slot[lane] : 0;
    warp_list_insert32<R>(v, cand, lane);
  }

  warp_list_store<R>(v, lists + warp * KP, lane);
  __syncthreads();
#pragma unroll
  for (int step = 1; step < NW; step <<= 1) {
    if ((warp % (2 * step)) == 0 && warp + step < NW) {
      warp_list_merge_from<R>(v, lists + (warp + step) * KP, lane);
      warp_list_store<R>(v, lists + warp * KP, lane);
    }
    __syncthreads();
  }
  if (warp == 0 && in_bounds(partials_cap == 0 || (static_cast<size_t>(blockIdx.x) + 1) * KP <= partials_cap, err))
    warp_list_store<R>(v, partials + static_cast<size_t>(blockIdx.x) * KP, lane);
}

// Streaming variant for large arrays: the same per-warp selection, with the
// 16-byte aligned body moved HBM -> shared memory by one-dimensional bulk
// copies (TMA) into a 3-stage ring of 64 KB tiles claimed dynamically from a
// global counter, so no registers are tied up by loads in flight. Sixteen
// consumer warps scan each tile; one producer warp feeds the ring.
//
// Before the first tile each CTA takes a lower bound on the final K-th key
// from its own slice of 32,768 values: the K-th largest of 256 group maxima
// (groups of 128 values). K distinct groups each hold a key at least that
// large, so at least K keys of the array are >= it and no key below it can be
// in the top K. The consumers read the slice while the producer fills the
// ring, and every key below the bound is dropped from the start. No CTA ever
// waits for another.
constexpr int kSW = 16;                         // consumer warps
constexpr int kSThreads = (kSW + 1) * 32;
constexpr int kSStages = 3;
constexpr int kSTileVec = 4096;                 // int4 per tile (64 KB)
constexpr int kSTileBytes = kSTileVec * 16;
constexpr int kBoundGroups = 256;               // group maxima per slice (K <= 256)
constexpr int kBoundSliceVec = 2 * kSTileVec;   // int4 per slice (32,768 values)
constexpr int kBoundVecPerThread = kBoundSliceVec / (kSW * 32);  // 16 int4 = 64 values per thread
static_assert(kSW * 32 == 2 * kBoundGroups, "two consumer threads per group");
static_assert(kBoundVecPerThread % 8 == 0, "slice loads go in batches of 8");

struct StreamParams {
  const int32_t* data;
  int64_t n;
  int k;
  uint64_t* partials;
  const uint64_t* theta0;  // optional: a lower bound on the K-th key (keys >= it are kept)
  unsigned* counters;  // [0] tile claims, [1] finished CTAs; zero between launches
  int* err;
  uint64_t timeout_ns;
  // Merge in the last CTA (when out_val is set): the K values and positions,
  // and the per-call error word handed to result_err / err_sticky.
  int32_t* out_val;
  int64_t* out_pos;
  int* err_sticky;
  int* result_err;
  size_t partials_cap;  // keys (checked builds; 0: not checked)
  int host_result;      // 1: results in mapped host memory, the host waits on result_err
};

// The last CTA merges in the ring's shared memory (the barriers after it are
// left alone).
constexpr int kMergeSmemBytes = kSStages * kSTileBytes;
constexpr int kMergeStageKeys = (kMergeSmemBytes / 8 - mergecore::kSurvivorCap - 2) & ~1;

__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kSW * 32) : "memory"); }

template <int KP>
__global__ void __launch_bounds__(kSThreads, 1) topk_i32_stream_kernel(const StreamParams p) {
  constexpr int R = KP / 32;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kSStages * kSTileBytes);
  uint64_t* empty = full + kSStages;
  int64_t* hdr_v0 = reinterpret_cast<int64_t*>(empty + kSStages);
  int* hdr_nv = reinterpret_cast<int*>(hdr_v0 + kSStages);
  WarpBuffer* bufs = reinterpret_cast<WarpBuffer*>(smem + kSStages * kSTileBytes + kSStages * 32);
  __shared__ int abort_flag;
  __shared__ uint64_t s_bound;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  pdl_launch_dependents();

  const uintptr_t addr = reinterpret_cast<uintptr_t>(p.data);
  int64_t head = static_cast<int64_t>(((16 - (addr & 15)) & 15) >> 2);
  if (head > p.n) head = p.n;
  const int64_t nvec = (p.n - head) >> 2;
  const int64_t tail0 = head + nvec * 4;
  const int4* vec = reinterpret_cast<const int4*>(p.data + head);
  const int64_t total_tiles = (nvec + kSTileVec - 1) / kSTileVec;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    s_bound = 0;
    for (int s = 0; s < kSStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kSW);
    }
    fence_mbar_init();
  }
  // Launched as a programmatic dependent: resident early, but the array, the
  // counters and the lists are touched only after the previous kernel on the
  // stream has finished.
  pdl_wait();
  __syncthreads();

  uint64_t v[R];
  warp_list_clear<R>(v);

  if (warp == kSW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      int64_t claim = static_cast<int64_t>(atomicAdd(&p.counters[0], 1u));
      int64_t issued = 0;
      bool aborted = false;
      for (int64_t i = 0;; ++i) {
        const int s = static_cast<int>(i % kSStages);
        const uint32_t u = static_cast<uint32_t>(i / kSStages);
        const bool end = claim >= total_tiles;
        int64_t v0 = 0;
        int nv = 0;
        if (!end) {
          v0 = claim * kSTileVec;
          nv = static_cast<int>(nvec - v0 < kSTileVec ? nvec - v0 : kSTileVec);
          claim = static_cast<int64_t>(atomicAdd(&p.counters[0], 1u));
        }
        if (u > 0 && !mbar_wait(&empty[s], (u - 1) & 1u, p.timeout_ns)) {
          atomicOr(p.err, kErrProducerTimeout);
          aborted = true;
          break;
        }
        if (*reinterpret_cast<volatile int*>(&abort_flag)) {
          aborted = true;
          break;
        }
        if (end) {
          hdr_nv[s] = -1;
          mbar_arrive(&full[s]);
          break;
        }
        hdr_v0[s] = v0;
        hdr_nv[s] = nv;
        mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(nv) * 16u);
        bulk_copy_g2s(ring + static_cast<size_t>(s) * kSTileBytes, vec + v0, static_cast<uint32_t>(nv) * 16u,
                      &full[s], pol);
        ++issued;
      }
      if (aborted) {
        abort_flag = 1;
        for (int64_t i = (issued > kSStages ? issued - kSStages : 0); i < issued; ++i) {
          const int s = static_cast<int>(i % kSStages);
          if (!mbar_wait(&full[s], static_cast<uint32_t>(i / kSStages) & 1u, p.timeout_ns))
            atomicOr(p.err, kErrDrainTimeout);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers
    WarpBuffer& buf = bufs[warp];
    uint64_t floor_key = 0;
    if (p.theta0) {
      const uint64_t b0 = *p.theta0;
      floor_key = b0 > 0 ? b0 - 1 : 0;
    }
    const int64_t slice = static_cast<int64_t>(blockIdx.x) * kBoundSliceVec;
    if (slice + kBoundSliceVec <= nvec) {  // CTA-uniform: every consumer warp takes part
      // Group g = threadIdx.x / 2 covers 32 vectors of the slice, 16 per
      // thread, strided by 512 vectors so that every load is coalesced (eight
      // loads in flight at a time).
      uint64_t best = 0;
#pragma unroll
      for (int j0 = 0; j0 < kBoundVecPerThread; j0 += 8) {
        int4 x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = __ldcg(vec + slice + threadIdx.x + (j0 + j) * (kSW * 32));
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t p0 = static_cast<uint32_t>(head + (slice + threadIdx.x + (j0 + j) * (kSW * 32)) * 4);
          best = umax64(best, make_ikey(x[j].x, p0));
          best = umax64(best, make_ikey(x[j].y, p0 + 1));
          best = umax64(best, make_ikey(x[j].z, p0 + 2));
          best = umax64(best, make_ikey(x[j].w, p0 + 3));
        }
      }
      best = umax64(best, shfl_xor_u64(best, 1));
      uint64_t* gmax = reinterpret_cast<uint64_t*>(bufs);  // 256 keys, 2 KB
      if ((threadIdx.x & 1) == 0) gmax[threadIdx.x >> 1] = best;
      consumer_bar();
      // The K-th largest group maximum is the one with exactly K-1 larger
      // (keys are distinct); each of the pair counts over half of the groups.
      const int h = threadIdx.x & 1;
      const ulonglong2* half = reinterpret_cast<const ulonglong2*>(gmax + h * (kBoundGroups / 2));
      int greater = 0;
#pragma unroll 8
      for (int j = 0; j < kBoundGroups / 4; ++j) {
        const ulonglong2 g = half[j];
        greater += (g.x > best ? 1 : 0) + (g.y > best ? 1 : 0);
      }
      greater += __shfl_xor_sync(kFullMask, greater, 1);
      if (h == 0 && greater == p.k - 1) s_bound = best;
      consumer_bar();  // also: every read of gmax is done before the buffers are reused
      const uint64_t b0 = s_bound;
      if (b0 > 1) floor_key = umax64(floor_key, b0 - 1);
    }
    uint64_t theta = floor_key;
    int cnt = 0;
    for (int64_t i = 0;; ++i) {
      const int s = static_cast<int>(i % kSStages);
      const uint32_t u = static_cast<uint32_t>(i / kSStages);
      if (!__all_sync(kFullMask, mbar_wait(&full[s], u & 1u, p.timeout_ns))) {
        if (lane == 0) atomicOr(p.err, kErrConsumerTimeout);
        abort_flag = 1;
        break;
      }
      const int nv = hdr_nv[s];
      if (nv < 0 || *reinterpret_cast<volatile int*>(&abort_flag)) break;
      const int64_t v0 = hdr_v0[s];
      const int4* tile = reinterpret_cast<const int4*>(ring + static_cast<size_t>(s) * kSTileBytes);
      // Each warp scans 4 x 32 consecutive int4 at a time (512 values).
      for (int c = warp * 128; c < nv; c += kSW * 128) {
        int4 x[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int t = c + q * 32 + lane;
          x[q] = (t < nv) ? tile[t] : make_int4(INT32_MIN, INT32_MIN, INT32_MIN, INT32_MIN);
        }
        bool in[4];
        uint32_t pos[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int t = c + q * 32 + lane;
          in[q] = t < nv;
          pos[q] = static_cast<uint32_t>(head + (v0 + t) * 4);
        }
        scan16<R>(v, buf, cnt, theta, floor_key, p.k, x, in, pos, lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (blockIdx.x == 0 && warp == 0) {
      // Unaligned head and the tail: at most 3 + 3 elements.
      const int64_t extra = head + (p.n - tail0);
      for (int64_t b = 0; b < extra; b += 32) {
        const int64_t t = b + lane;
        const bool in = t < extra;
        int64_t pos = 0;
        if (in) pos = (t < head) ? t : tail0 + (t - head);
        const uint64_t key = in ? make_ikey(p.data[pos], static_cast<uint32_t>(pos)) : 0;
        offer<R>(v, buf, cnt, theta, floor_key, p.k, key, in && key > theta, lane);
      }
    }
    if (cnt > 0) {
      const uint64_t cand = (lane < cnt) ? buf.slot[lane] : 0;
      warp_list_insert32<R>(v, cand, lane);
    }
  }

  // CTA merge of the consumer warps' lists (reusing the ring).
  __syncthreads();
  uint64_t* lists = reinterpret_cast<uint64_t*>(smem);
  if (warp < kSW) warp_list_store<R>(v, lists + warp * KP, lane);
  __syncthreads();
#pragma unroll
  for (int step = 1; step < kSW; step <<= 1) {
    if (warp < kSW && (warp % (2 * step)) == 0 && warp + step < kSW) {
      warp_list_merge_from<R>(v, lists + (warp + step) * KP, lane);
      warp_list_store<R>(v, lists + warp * KP, lane);
    }
    __syncthreads();
  }
  if (warp == 0 &&
      in_bounds(p.partials_cap == 0 || (static_cast<size_t>(blockIdx.x) + 1) * KP <= p.partials_cap, p.err))
    warp_list_store<R>(v, p.partials + static_cast<size_t>(blockIdx.x) * KP, lane);
  __shared__ int s_last;
  __threadfence();  // this CTA's list is visible before its ticket
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned done = atomicAdd(&p.counters[1], 1u);
    s_last = done == gridDim.x - 1 ? 1 : 0;
    if (s_last) {
      atomicExch(&p.counters[0], 0u);
      atomicExch(&p.counters[1], 0u);
    }
  }
  __syncthreads();
  if (s_last && p.out_val) {
    // Stage 2 in the last CTA to finish: every other CTA's list is written.
    __threadfence();
    mergecore::MergeOut o;
    o.k = p.k;
    o.int_keys = 1;
    o.out_a = p.out_val;
    o.out_b = p.out_pos;
    o.kth_out = nullptr;
    o.q = 0;
    o.stride = KP;
    o.lens = nullptr;
    o.region = static_cast<size_t>(gridDim.x) * KP;
    o.err = p.err;
    mergecore::merge_lists<KP, kSThreads>(o, p.partials, static_cast<int>(gridDim.x),
                                          reinterpret_cast<uint64_t*>(smem), kMergeSmemBytes, kMergeStageKeys);
    // Hand the per-call error word to the sticky word and re-arm it, then
    // publish it to the host-visible result after the results.
    __shared__ int s_err;
    if (threadIdx.x == 0) {
      const int e = atomicOr(p.err, 0);
      if (e && p.err_sticky) atomicOr(p.err_sticky, e);
      atomicExch(p.err, 0);
      s_err = e;
    }
    __syncthreads();
    publish_result_word(p.result_err, s_err, p.host_result != 0);
  }
}

constexpr int kStreamSmem = kSStages * kSTileBytes + kSStages * 32 + kSW * static_cast<int>(sizeof(WarpBuffer));

template <int KP>
cudaError_t launch_stream_t(const StreamParams& p, int grid, cudaStream_t stream) {
  auto fn = topk_i32_stream_kernel<KP>;
  static PerDeviceOnce once;
  const cudaError_t limit =
      once.run([fn] { return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kStreamSmem); });
  if (limit != cudaSuccess) return limit;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kSThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(kStreamSmem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, p);
}

// Wait on an mbarrier nothing ever arrives at, through the library's bounded
// wait, and report the timeout. Exercises the timeout path without a fault.
__global__ void wait_probe_kernel(int* err, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, timeout_ns)) atomicOr(err, kErrProbeTimeout);
}

template <int KP>
cudaError_t launch_t(const I32Launch& a, cudaStream_t stream) {
  topk_i32_stage1_kernel<KP><<<a.grid, NW * 32, 0, stream>>>(a.data, a.n, a.k, a.partials, a.theta0, a.partials_cap,
                                                              a.err);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_topk_i32_stage1(const I32Launch& a, cudaStream_t stream) {
  switch (list_width(a.k)) {
    case 32: return launch_t<32>(a, stream);
    case 64: return launch_t<64>(a, stream);
    case 128: return launch_t<128>(a, stream);
    case 256: return launch_t<256>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_topk_i32_stream(const I32StreamLaunch& a, cudaStream_t stream) {
  StreamParams p;
  p.data = a.data;
  p.n = a.n;
  p.k = a.k;
  p.partials = a.partials;
  p.theta0 = a.theta0;
  p.counters = a.counters;
  p.err = a.err;
  p.timeout_ns = a.timeout_ns;
  p.out_val = a.out_val;
  p.host_result = a.host_result;
  p.out_pos = a.out_pos;
  p.err_sticky = a.err_sticky;
  p.result_err = a.result_err;
  p.partials_cap = a.partials_cap;
  if (a.k < 1 || a.k > kBoundGroups) return cudaErrorInvalidValue;
  switch (list_width(a.k)) {
    case 32: return launch_stream_t<32>(p, a.grid, stream);
    case 64: return launch_stream_t<64>(p, a.grid, stream);
    case 128: return launch_stream_t<128>(p, a.grid, stream);
    case 256: return launch_stream_t<256>(p, a.grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_wait_probe(int* err, uint64_t timeout_ns, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace rbf
