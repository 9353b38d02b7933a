// merge.cu -- global top-K from per-CTA best-first lists, one CTA per query.
//
// The merge step of GPU-Resident Top-K for Agentic RAG (section 4 step 4:
// combine the per-block lists into the global top-K, best first, with the
// lower index winning exact ties) and stage 2 of the two-stage int32 top-K
// (CUDA programming model series 9, section 3.1: one block over the GRID x K
// stage-1 candidates).
//
// Each of the CTA's 32 warps folds a strided subset of the lists into a
// register bitonic list (reversed max + bitonic merge per list), then the warp
// lists are merged pairwise in shared memory, five levels, and warp 0 writes
// the best K decoded. The keys already encode the ordering rule, so every
// comparison is one unsigned 64-bit compare.
#include "rbf_device.cuh"
#include "rbf_internal.h"

namespace rbf {
namespace {

constexpr int kMergeWarps = 32;

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
};

template <int KP>
__global__ void __launch_bounds__(kMergeWarps * 32, 1) merge_partials_kernel(const Params p) {
  constexpr int R = KP / 32;
  extern __shared__ __align__(16) uint64_t lists[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t* base = p.partials + static_cast<size_t>(blockIdx.x) * p.lists * KP;

  uint64_t v[R];
  warp_list_clear<R>(v);
  for (int l = warp; l < p.lists; l += kMergeWarps) warp_list_merge_from<R>(v, base + static_cast<size_t>(l) * KP, lane);
  warp_list_store<R>(v, lists + warp * KP, lane);
  __syncthreads();
#pragma unroll
  for (int step = 1; step < kMergeWarps; step <<= 1) {
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

template <int KP>
cudaError_t launch_t(const Params& p, int queries, cudaStream_t stream) {
  auto fn = merge_partials_kernel<KP>;
  const int smem = kMergeWarps * KP * 8;
  static int configured = 0;
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  fn<<<queries, kMergeWarps * 32, smem, stream>>>(p);
  return cudaGetLastError();
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
  switch (list_width(a.k)) {
    case 32: return launch_t<32>(p, a.queries, stream);
    case 64: return launch_t<64>(p, a.queries, stream);
    case 128: return launch_t<128>(p, a.queries, stream);
    case 256: return launch_t<256>(p, a.queries, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace rbf
