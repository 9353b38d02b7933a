// merge.cu -- global top-K from per-CTA best-first lists, one CTA per query.
//
// The merge step of GPU-Resident Top-K for Agentic RAG (section 4 step 4:
// combine the per-block lists into the global top-K, best first, with the
// lower index winning exact ties) and stage 2 of the two-stage int32 top-K
// (CUDA programming model series 9, section 3.1: one block over the GRID x K
// stage-1 candidates).
//
// The first K keys of every list (nothing past a list's K-th entry can reach
// the global top-K) are staged in shared memory by all threads at once, one
// round trip to L2; each warp then folds a strided subset of the staged lists
// into a register bitonic list (reversed max + bitonic merge per list). The warp
// lists are then merged pairwise in shared memory and warp 0 writes the best
// K decoded. The keys already encode the ordering rule, so every comparison
// is one unsigned 64-bit compare. The kernel is launched as a programmatic
// dependent of the kernel that wrote the lists, so its launch overlaps that
// kernel's tail; it waits for the lists before touching them.
#include <algorithm>

#include "rbf_device.cuh"
#include "rbf_internal.h"

namespace rbf {
namespace {

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
  int stage_lists;    // lists staged in shared memory at a time
};

template <int KP, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, 1) merge_partials_kernel(const Params p) {
  constexpr int R = KP / 32;
  extern __shared__ __align__(16) uint64_t smem[];
  uint64_t* lists = smem;                          // WARPS lists of KP keys (the tree)
  uint64_t* stage = smem + WARPS * KP;             // staged list heads, k keys each
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  pdl_wait();
  const uint64_t* base = p.partials + static_cast<size_t>(blockIdx.x) * p.lists * KP;

  uint64_t v[R];
  warp_list_clear<R>(v);
  // Lists are staged in groups that fit the staging area: every thread loads
  // its share of the group's first-k keys at once (one round trip to L2),
  // then each warp folds a strided subset of the staged lists.
  const int per_group = p.stage_lists;
  for (int g0 = 0; g0 < p.lists; g0 += per_group) {
    const int gl = min(per_group, p.lists - g0);
    const int total = gl * p.k;
    for (int i = threadIdx.x; i < total; i += WARPS * 32) {
      const int l = i / p.k;
      const int e = i - l * p.k;
      stage[i] = __ldcg(base + static_cast<size_t>(g0 + l) * KP + e);
    }
    __syncthreads();
    for (int l = warp; l < gl; l += WARPS) {
      const uint64_t* src = stage + l * p.k;
#pragma unroll
      for (int s = 0; s < R; ++s) {
        const int e = KP - 1 - (s * 32 + lane);
        v[s] = umax64(v[s], e < p.k ? src[e] : 0ull);
      }
      warp_bitonic_merge_desc<R>(v, lane);
    }
    __syncthreads();
  }
  warp_list_store<R>(v, lists + warp * KP, lane);
  __syncthreads();
#pragma unroll
  for (int step = 1; step < WARPS; step <<= 1) {
    if ((warp % (2 * step)) == 0) {
      warp_list_merge_from<R>(v, lists + (warp + step) * KP, lane);
      warp_list_store<R>(v, lists + warp * KP, lane);
    }
    __syncthreads();
  }
  if (warp == 0) {
#pragma unroll
    for (int s = 0; s < R; ++s) {
      const int e = s * 32 + lane;
      if (p.kth_out && e == p.k - 1) p.kth_out[blockIdx.x] = v[s];
      if (e < p.k) {
        const size_t o = static_cast<size_t>(blockIdx.x) * p.k + e;
        if (p.int_keys) {
          p.out_a[o] = ikey_value(v[s]);
          static_cast<int64_t*>(p.out_b)[o] = static_cast<int64_t>(key_index(v[s]));
        } else {
          p.out_a[o] = static_cast<int32_t>(key_index(v[s]));
          static_cast<float*>(p.out_b)[o] = key_score(v[s]);
        }
      }
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.err_call) {
    // Hand the per-call device error word to the host-visible result and
    // the sticky word, then re-arm it for the next call.
    const int e = *p.err_call;
    if (p.result_err) *p.result_err = e;
    if (e && p.err_sticky) atomicOr(p.err_sticky, e);
    *p.err_call = 0;
  }
}

constexpr int kStageBytes = 160 * 1024;  // shared memory for staged list heads

template <int KP, int WARPS>
cudaError_t launch_t(Params p, int queries, cudaStream_t stream) {
  auto fn = merge_partials_kernel<KP, WARPS>;
  p.stage_lists = std::max(1, std::min(p.lists, kStageBytes / (8 * p.k)));
  const int smem = WARPS * KP * 8 + p.stage_lists * p.k * 8;
  static int configured = 0;
  const int want = WARPS * KP * 8 + kStageBytes;
  if (want > configured) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
    if (e != cudaSuccess) return e;
    configured = want;
  }
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

}  // namespace

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
  switch (list_width(a.k)) {
    case 32: return launch_t<32, 32>(p, a.queries, stream);
    case 64: return launch_t<64, 32>(p, a.queries, stream);
    case 128: return launch_t<128, 32>(p, a.queries, stream);
    case 256: return launch_t<256, 16>(p, a.queries, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace rbf
