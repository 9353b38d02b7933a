// merge.cu -- global top-K from per-CTA best-first lists, one CTA per query.
//
// The merge step of GPU-Resident Top-K for Agentic RAG (section 4 step 4) and
// stage 2 of the two-stage int32 top-K (CUDA programming model series 9,
// section 3.1); the per-query work is in merge_core.cuh. The kernel is
// launched as a programmatic dependent of the kernel that wrote the lists,
// so its launch overlaps that kernel's tail; it waits for the lists before
// touching them.
#include <algorithm>

#include "merge_core.cuh"
#include "rbf_device.cuh"
#include "rbf_internal.h"

namespace rbf {
namespace {

using mergecore::fast_smem_bytes;
using mergecore::kSurvivorCap;
using mergecore::MergeOut;

struct Params {
  const uint64_t* partials;
  int lists;
  int k;
  int int_keys;
  int32_t* out_a;
  void* out_b;
  int* err_call;
  int* err_sticky;
  int* result_err;
  uint64_t* kth_out;  // optional: the K-th key of each query
  int smem_bytes;     // dynamic shared memory of the launch
  int stride;         // keys from one list to the next
  const int* lens;    // optional: [query][list] valid keys per list
  int stage_keys;     // shared-memory budget (keys) for staged list heads
  size_t partials_cap;  // keys (checked builds; 0: not checked)
  int host_result;      // 1: one query, results in mapped host memory, the host waits on result_err
};

constexpr int kManyQueries = 64;          // from this many queries on, merge CTAs are 8 warps
constexpr int kStageBytes = 160 * 1024;   // shared memory for staged list heads (at most)
constexpr int kStageKeys = kStageBytes / 8;

template <int KP, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, 1) merge_partials_kernel(const Params p) {
  extern __shared__ __align__(16) uint64_t smem[];
  pdl_launch_dependents();  // a following scoring pass may start streaming; it waits before using our output
  pdl_wait();
  const uint64_t* base = p.partials + static_cast<size_t>(blockIdx.x) * p.lists * p.stride;
  MergeOut o;
  o.k = p.k;
  o.int_keys = p.int_keys;
  o.out_a = p.out_a;
  o.out_b = p.out_b;
  o.kth_out = p.kth_out;
  o.q = blockIdx.x;
  o.stride = p.stride;
  o.lens = p.lens ? p.lens + static_cast<size_t>(blockIdx.x) * p.lists : nullptr;
  if (p.partials_cap) {
    const size_t off = static_cast<size_t>(blockIdx.x) * p.lists * p.stride;
    o.region = p.partials_cap > off ? p.partials_cap - off : 1;  // 1: every read is out of bounds
  }
  o.err = p.err_sticky ? p.err_sticky : p.err_call;
  mergecore::merge_lists<KP, WARPS * 32>(o, base, p.lists, smem, p.smem_bytes, p.stage_keys);
  if (!p.err_call) return;
  // Hand the per-call device error word to the sticky word and re-arm it;
  // the result word follows the results. With one query (one CTA) the word
  // is published after this CTA's results, so a host caller may wait for
  // it; with several, only the stream's completion covers every CTA.
  __shared__ int s_err;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const int e = *p.err_call;
    if (e && p.err_sticky) atomicOr(p.err_sticky, e);
    *p.err_call = 0;
    s_err = e;
  }
  if (gridDim.x == 1) {
    __syncthreads();
    publish_result_word(p.result_err, s_err, p.host_result != 0);
  } else if (blockIdx.x == 0 && threadIdx.x == 0 && p.result_err) {
    *p.result_err = s_err;
  }
}

template <int KP, int WARPS>
cudaError_t launch_t(Params p, int queries, cudaStream_t stream) {
  auto fn = merge_partials_kernel<KP, WARPS>;
  const int stage_lists = std::max(1, std::min(p.lists, p.stage_keys / p.k));
  const int smem =
      std::max(WARPS * KP * 8 + stage_lists * p.k * 8, fast_smem_bytes(p.lists, p.k, p.stage_keys));
  p.smem_bytes = smem;
  // The largest launch of this instance, set once per device.
  static PerDeviceOnce once;
  const cudaError_t limit = once.run([fn] {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                WARPS * KP * 8 + kStageBytes + (kSurvivorCap + 2) * 8);
  });
  if (limit != cudaSuccess) return limit;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(queries));
  cfg.blockDim = dim3(WARPS * 32);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, p);
}

// Row-sharded search (GPU-Resident Top-K for Agentic RAG, section 4 step 1
// and section 9: a corpus beyond one GPU is split into row shards): each
// shard's best-first (global index, score) list of one query becomes a list
// of keys with the same ordering rule, so that the merge kernel can combine
// the shards' lists like the per-CTA lists of one search. Output slot
// [q][s][e] takes input [s][q][e]; missing entries (index < 0) and the
// slots from k to kp are the empty key.
__global__ void encode_shard_lists_kernel(const int32_t* __restrict__ idx, const float* __restrict__ score, int g,
                                          int b, int k, int kp, uint64_t* __restrict__ out) {
  pdl_launch_dependents();  // the merge may be scheduled now; it waits for these keys
  const int64_t total = static_cast<int64_t>(b) * g * kp;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int e = static_cast<int>(i % kp);
    const int64_t r = i / kp;
    const int s = static_cast<int>(r % g);
    const int64_t q = r / g;
    uint64_t key = 0;
    if (e < k) {
      const int64_t src = (static_cast<int64_t>(s) * b + q) * k + e;
      const int32_t ix = idx[src];
      if (ix >= 0) key = make_key(score[src], static_cast<uint32_t>(ix));
    }
    out[i] = key;
  }
}

// The batched path's bound: one warp per query over its `total` keys (the
// pre-pass lists, contiguous per query). The warp finds the largest score code
// c (the key's high word) that at least K of the keys reach, one bit at a time
// from the top: a bit is kept when K keys still reach the code with it set.
// K distinct rows then score at least c, so c << 32 (index word zero) bounds
// the K-th key from below; 0 if fewer than K keys are nonzero. A CTA of two
// such warps without shared memory fits beside a scoring CTA on its SM, and
// 128 of them cover 256 queries, one per SM beside the pre-pass: the main
// pass's CTAs never wait for these to leave.
// PL keys per lane (PL * 32 >= total); the per-bit count runs in four
// independent sums so that it is not one long chain of dependent adds.
constexpr int kKthWarpsPerCta = 2;

template <int PL>
__global__ void __launch_bounds__(kKthWarpsPerCta * 32) kth_code_kernel(const uint64_t* __restrict__ keys,
                                                                        int queries, int total, int k,
                                                                        uint64_t* __restrict__ kth_out) {
  static_assert(PL % 4 == 0 && PL * 32 <= RBF_KTH_MAX_KEYS, "keys per lane");
  pdl_launch_dependents();  // the main pass may be scheduled now; it waits for the bounds
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int q = blockIdx.x * kKthWarpsPerCta + (threadIdx.x >> 5);
  if (q >= queries) return;
  const uint64_t* src = keys + static_cast<size_t>(q) * total;
  uint32_t c[PL];
#pragma unroll
  for (int j = 0; j < PL; ++j) {
    const int i = j * 32 + lane;
    c[j] = i < total ? static_cast<uint32_t>(__ldcg(src + i) >> 32) : 0u;
  }
  uint32_t res = 0;
#pragma unroll 1
  for (int bit = 31; bit >= 0; --bit) {
    const uint32_t t = res | (1u << bit);
    unsigned n[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int j = 0; j < PL; ++j) n[j & 3] += c[j] >= t ? 1u : 0u;
    if (__reduce_add_sync(0xffffffffu, (n[0] + n[1]) + (n[2] + n[3])) >= static_cast<unsigned>(k)) res = t;
  }
  if (lane == 0) kth_out[q] = static_cast<uint64_t>(res) << 32;
}

}  // namespace

cudaError_t launch_kth_of_lists(const uint64_t* keys, int queries, int total, int k, uint64_t* kth_out,
                                cudaStream_t stream) {
  if (queries < 1 || total < 1 || total > RBF_KTH_MAX_KEYS || k < 1 || k > RBF_KTH_MAX_K) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((queries + kKthWarpsPerCta - 1) / kKthWarpsPerCta));
  cfg.blockDim = dim3(kKthWarpsPerCta * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int per_lane = (total + 31) / 32;
  if (per_lane <= 8) return cudaLaunchKernelEx(&cfg, kth_code_kernel<8>, keys, queries, total, k, kth_out);
  if (per_lane <= 16) return cudaLaunchKernelEx(&cfg, kth_code_kernel<16>, keys, queries, total, k, kth_out);
  if (per_lane <= 24) return cudaLaunchKernelEx(&cfg, kth_code_kernel<24>, keys, queries, total, k, kth_out);
  return cudaLaunchKernelEx(&cfg, kth_code_kernel<32>, keys, queries, total, k, kth_out);
}

cudaError_t launch_encode_shard_lists(const int32_t* idx, const float* score, int g, int b, int k, int kp,
                                      uint64_t* out, int num_sms, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(b) * g * kp;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, static_cast<int64_t>(num_sms) * 8);
  encode_shard_lists_kernel<<<static_cast<unsigned>(std::max<int64_t>(1, blocks)), 256, 0, stream>>>(idx, score, g,
                                                                                                     b, k, kp, out);
  return cudaGetLastError();
}

cudaError_t launch_merge(const MergeLaunch& a, cudaStream_t stream) {
  Params p;
  p.partials = a.partials;
  p.lists = a.lists;
  p.k = a.k;
  p.int_keys = a.int_keys;
  p.out_a = a.out_a;
  p.out_b = a.out_b;
  p.err_call = a.err_call;
  p.err_sticky = a.err_sticky;
  p.result_err = a.result_err;
  p.kth_out = a.kth_out;
  p.stride = a.stride > 0 ? a.stride : list_width(a.k);
  p.lens = a.lens;
  p.partials_cap = a.partials_cap;
  p.host_result = a.host_result;
  // Short lists (a prefix of K valid keys, or fewer): stage 32 keys of each
  // (the rest is read from L2 if it survives), so that the CTA's shared
  // memory stays small and all queries run in one wave.
  p.stage_keys = a.short_lists ? std::min(kStageKeys, std::max(2 * a.k, a.lists * 32)) : kStageKeys;
  // One query: a wide CTA to shorten the single merge. Many queries: 8-warp
  // CTAs, so that several fit on each SM and all queries run in one wave.
  if (a.queries >= kManyQueries) {
    switch (list_width(a.k)) {
      case 32: return launch_t<32, 8>(p, a.queries, stream);
      case 64: return launch_t<64, 8>(p, a.queries, stream);
      case 128: return launch_t<128, 8>(p, a.queries, stream);
      case 256: return launch_t<256, 8>(p, a.queries, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (list_width(a.k)) {
    case 32: return launch_t<32, 32>(p, a.queries, stream);
    case 64: return launch_t<64, 32>(p, a.queries, stream);
    case 128: return launch_t<128, 32>(p, a.queries, stream);
    case 256: return launch_t<256, 16>(p, a.queries, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace rbf
