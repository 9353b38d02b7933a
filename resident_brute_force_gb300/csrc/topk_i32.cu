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

template <int KP>
__global__ void __launch_bounds__(NW * 32) topk_i32_stage1_kernel(const int32_t* __restrict__ data, int64_t n,
                                                                  int k, uint64_t* partials,
                                                                  const uint64_t* __restrict__ theta0) {
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
    // Cheap superset test first: a key can only beat theta if its value code
    // is at least theta's. Most steps end here with one vote.
    const uint32_t theta_hi = static_cast<uint32_t>(theta >> 32);
    bool maybe = false;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const bool in = c + u * 32 + lane < v1;
      maybe |= in && ((static_cast<uint32_t>(x[u].x) ^ 0x80000000u) >= theta_hi);
      maybe |= in && ((static_cast<uint32_t>(x[u].y) ^ 0x80000000u) >= theta_hi);
      maybe |= in && ((static_cast<uint32_t>(x[u].z) ^ 0x80000000u) >= theta_hi);
      maybe |= in && ((static_cast<uint32_t>(x[u].w) ^ 0x80000000u) >= theta_hi);
    }
    if (!__any_sync(kFullMask, maybe)) continue;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = c + u * 32 + lane;
      const bool in = i < v1;
      const uint32_t pos = static_cast<uint32_t>(head + i * 4);
      const int32_t e[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint64_t key = make_ikey(e[j], pos + j);
        offer<R>(v, buf, cnt, theta, floor_key, k, key, in && key > theta, lane);
      }
    }
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
  if (warp == 0) warp_list_store<R>(v, partials + static_cast<size_t>(blockIdx.x) * KP, lane);
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
  topk_i32_stage1_kernel<KP><<<a.grid, NW * 32, 0, stream>>>(a.data, a.n, a.k, a.partials, a.theta0);
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

cudaError_t launch_wait_probe(int* err, uint64_t timeout_ns, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace rbf
