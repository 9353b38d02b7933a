// merge.cu -- global top-K from per-CTA best-first lists, one CTA per query.
//
// The merge step of GPU-Resident Top-K for Agentic RAG (section 4 step 4:
// combine the per-block lists into the global top-K, best first, with the
// lower index winning exact ties) and stage 2 of the two-stage int32 top-K
// (CUDA programming model series 9, section 3.1: one block over the GRID x K
// stage-1 candidates).
//
// Each warp folds a strided subset of the lists into a register bitonic list
// (reversed max + bitonic merge per list), loading the next list while it
// merges the current one and reading only the first K entries of each list
// (nothing past a list's K-th entry can reach the global top-K). The warp
// lists are then merged pairwise in shared memory and warp 0 writes the best
// K decoded. The keys already encode the ordering rule, so every comparison
// is one unsigned 64-bit compare. The kernel is launched as a programmatic
// dependent of the kernel that wrote the lists, so its launch overlaps that
// kernel's tail; it waits for the lists before touching them.
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
};

// List l's element KP-1-e for e = s*32 + lane, as the second operand of a
// reversed-max fold; entries past the K-th read as the empty sentinel.
template <int R>
__device__ __forceinline__ void load_reversed(uint64_t (&dst)[R], const uint64_t* list, int k, int lane) {
  constexpr int KP = 32 * R;
#pragma unroll
  for (int s = 0; s < R; ++s) {
    const int e = KP - 1 - (s * 32 + lane);
    dst[s] = (e < k) ? __ldcg(list + e) : 0ull;
  }
}

template <int KP, int WARPS>
__global__ void __launch_bounds__(WARPS * 32, 1) merge_partials_kernel(const Params p) {
  constexpr int R = KP / 32;
  extern __shared__ __align__(16) uint64_t lists[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  pdl_wait();
  const uint64_t* base = p.partials + static_cast<size_t>(blockIdx.x) * p.lists * KP;

  uint64_t v[R];
  warp_list_clear<R>(v);
  uint64_t nxt[R];
  int l = warp;
  if (l < p.lists) load_reversed<R>(nxt, base + static_cast<size_t>(l) * KP, p.k, lane);
  while (l < p.lists) {
    uint64_t cur[R];
#pragma unroll
    for (int s = 0; s < R; ++s) cur[s] = nxt[s];
    const int ln = l + WARPS;
    if (ln < p.lists) load_reversed<R>(nxt, base + static_cast<size_t>(ln) * KP, p.k, lane);
#pragma unroll
    for (int s = 0; s < R; ++s) v[s] = umax64(v[s], cur[s]);
    warp_bitonic_merge_desc<R>(v, lane);
    l = ln;
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

template <int KP, int WARPS>
cudaError_t launch_t(const Params& p, int queries, cudaStream_t stream) {
  auto fn = merge_partials_kernel<KP, WARPS>;
  const int smem = WARPS * KP * 8;
  static int configured = 0;
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = smem;
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
