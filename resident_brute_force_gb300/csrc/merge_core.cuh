// merge_core.cuh -- the merge of best-first key lists into one query's top-K,
// shared by the merge kernel and by kernels that merge their own per-CTA
// lists in their last CTA.
//
// The merge step of GPU-Resident Top-K for Agentic RAG (section 4 step 4:
// combine the per-block lists into the global top-K, best first, with the
// lower index winning exact ties) and stage 2 of the two-stage int32 top-K
// (CUDA programming model series 9, section 3.1: one block over the GRID x K
// stage-1 candidates).
//
// Fast path (the lists' first keys fit in shared memory). The first K keys of
// every list (nothing past a list's K-th entry can reach the global top-K)
// are staged in shared memory by all threads at once, one round trip to L2. A
// lower bound B on the global K-th key then comes from two rows of the staged
// lists: with t the smallest power of two for which m = ceil(K/t) is at most
// the number of lists, the m-th largest t-th key X (found by ranking each
// t-th key against warp-sorted runs of them) has m lists each holding t
// keys >= X, so at least K keys are >= X; and each list's K-th key is itself
// such a bound. Only the keys >= B can be in the answer (in each best-first
// list they form a prefix); they are gathered (one list per thread), and each
// one's place is the number of gathered keys greater than it (keys are
// distinct). On random data a few more than K keys survive. If more than
// kSurvivorCap survive, or there are too many lists, the general merge runs
// instead: the lists are staged
// in groups, each warp folds a strided subset of them into a register bitonic
// list (reversed max + bitonic merge per list), the warp lists are merged
// pairwise in shared memory and warp 0 writes the best K decoded.
//
// The keys already encode the ordering rule, so every comparison is one
// unsigned 64-bit compare.
#pragma once

#include "rbf_device.cuh"

namespace rbf {
namespace mergecore {

// Where one query's result goes: K entries at q*K of out_a / out_b (int32
// value + int64 position for integer keys, int32 index + fp32 score for score
// keys), and optionally the K-th key at kth_out[q]. The lists are `stride`
// keys apart; with `lens` list l holds lens[l] keys (entries past that are
// never read and count as empty), else all `stride`.
struct MergeOut {
  int k;
  int int_keys;
  int32_t* out_a;
  void* out_b;
  uint64_t* kth_out;
  size_t q;
  int stride;
  const int* lens;
  size_t region = 0;  // keys readable from the lists' base (checked builds; 0: not checked)
  int* err = nullptr; // where a checked build reports an index outside region
};

// Valid keys of list l.
__device__ __forceinline__ int list_len(const MergeOut& p, int l) { return p.lens ? p.lens[l] : p.stride; }

// Key e of list l, or the empty key past the list's end.
__device__ __forceinline__ uint64_t list_key(const MergeOut& p, const uint64_t* base, int l, int e) {
  const size_t off = static_cast<size_t>(l) * p.stride + e;
  return e < list_len(p, l) && in_bounds(p.region == 0 || off < p.region, p.err) ? __ldcg(base + off) : 0ull;
}

constexpr int kSurvivorCap = 2048;  // keys gathered by the fast path
constexpr int kFastMaxLists = 512;  // lists the bound selection handles (its work grows as lists^2 / 32)

__device__ __forceinline__ void emit(const MergeOut& p, int e, uint64_t key) {
  const size_t o = p.q * static_cast<size_t>(p.k) + e;
  if (p.int_keys) {
    p.out_a[o] = ikey_value(key);
    static_cast<int64_t*>(p.out_b)[o] = static_cast<int64_t>(key_index(key));
  } else {
    p.out_a[o] = static_cast<int32_t>(key_index(key));
    static_cast<float*>(p.out_b)[o] = key_score(key);
  }
  if (p.kth_out && e == p.k - 1) p.kth_out[p.q] = key;
}

// Copy the first k keys of lists [l0, l0 + count) to dst (list-major, k per
// list, empty keys past a list's end) with U loads in flight per thread
// before any is stored, so the copy costs one L2 round trip per U x threads
// keys (16 for CTAs of up to 256 threads, 8 for wider ones, which must stay
// within 64 registers).
template <int NT, int U = (NT <= 256 ? 16 : 8)>
__device__ __forceinline__ void stage_heads(const MergeOut& p, uint64_t* dst, const uint64_t* base, int l0, int count,
                                            int k) {
  const int total = count * k;
  for (int i0 = 0; i0 < total; i0 += U * NT) {
    uint64_t r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * NT + static_cast<int>(threadIdx.x);
      r[u] = 0;
      if (i < total) {
        const int l = i / k;
        r[u] = list_key(p, base, l0 + l, i - l * k);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * NT + static_cast<int>(threadIdx.x);
      if (i < total) dst[i] = r[u];
    }
  }
}

// The row t of the bound: the smallest power of two with ceil(K/t) <= lists,
// at most K.
__host__ __device__ constexpr int fast_row(int lists, int k) {
  int t = 1;
  while ((k + t - 1) / t > lists) t <<= 1;
  return t < k ? t : k;
}

// Keys of each list the fast path stages, given room for stage_keys keys:
// min(K, max(32, t)) if they fit (survivors rarely reach further into a
// list; those that do are read from L2), else the largest multiple of 32
// that does (at least 32); 0 if the fast path does not apply.
__host__ __device__ constexpr int fast_prefix(int lists, int k, int stage_keys) {
  if (lists > kFastMaxLists) return 0;
  const int t = fast_row(lists, k);
  const int want = k < (t > 32 ? t : 32) ? k : (t > 32 ? t : 32);
  return lists * want <= stage_keys ? want : (stage_keys / lists) & ~31;
}

// Shared memory (bytes) the fast path needs: the staged prefixes and the
// survivors; 0 if it does not apply.
__host__ __device__ constexpr int fast_smem_bytes(int lists, int k, int stage_keys) {
  return fast_prefix(lists, k, stage_keys) > 0
             ? (((lists * fast_prefix(lists, k, stage_keys) + 1) & ~1) + kSurvivorCap + 2) * 8
             : 0;
}

// Returns false (block-uniform) if the fast path does not apply; nothing has
// been written then.
template <int KP, int NT>
__device__ bool merge_fast(const MergeOut& p, const uint64_t* base, int L, uint64_t* smem, int stage_keys) {
  constexpr int WARPS = NT / 32;
  __shared__ unsigned long long s_bound;
  __shared__ int s_count;
  const int k = p.k;
  const int P = fast_prefix(L, k, stage_keys);  // staged keys per list
  if (P < 1 || (P < k && P < 32)) return false;
  const int t = fast_row(L, k);  // t = K gives m = 1, which every list count satisfies
  if (t > P) return false;
  const int m = (k + t - 1) / t;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  uint64_t* stage = smem;                      // L lists x P keys
  uint64_t* surv = smem + ((L * P + 1) & ~1);  // kSurvivorCap + 2 keys, 16-byte aligned
  if (tid == 0) {
    s_bound = 1;  // excludes the empty slots (key 0)
    s_count = 0;
  }
  stage_heads<NT>(p, stage, base, 0, L, P);
  __syncthreads();
  // The lists' t-th keys in runs of 32, each sorted best first by one warp
  // (they sit where the survivors go later; the last run is padded with the
  // empty key).
  uint64_t* row = surv;
  const int runs = (L + 31) >> 5;
  for (int r = warp; r < runs; r += WARPS) {
    const int l = r * 32 + lane;
    row[l] = warp_sort32_desc(l < L ? stage[l * P + t - 1] : 0ull, lane);
  }
  __syncthreads();

  // One list per thread: the number of lists whose t-th key beats this one's
  // is the sum over the runs of a 5-step binary search (keys are distinct,
  // except empty ones, which beat nothing).
  for (int l = tid; l < L; l += NT) {
    const uint64_t x = stage[l * P + t - 1];
    int greater = 0;
    for (int r = 0; r < runs; ++r) {
      const uint64_t* run = row + r * 32;
      int lo = 0;
#pragma unroll
      for (int step = 16; step > 0; step >>= 1) lo += run[lo + step - 1] > x ? step : 0;
      greater += lo + (run[lo] > x ? 1 : 0);
    }
    uint64_t b = k <= P ? stage[l * P + k - 1] : list_key(p, base, l, k - 1);
    if (greater == m - 1) b = umax64(b, x);
    atomicMax(&s_bound, static_cast<unsigned long long>(b));
  }
  __syncthreads();
  const uint64_t bound = s_bound;

  // Gather each list's prefix of keys >= bound (lists are best first, so
  // the prefix ends at the first key below it), one list per thread within
  // the staged keys: the thread counts its prefix, a warp scan turns the
  // counts into offsets behind one shared atomic per warp, and the thread
  // copies its keys. A prefix that runs past the staged keys (rare) is
  // continued from L2 by the whole warp, 32 keys per round trip.
  for (int l0 = 0; l0 < L; l0 += NT) {
    const int l = l0 + tid;
    const int lim = min(P, k);
    int c = 0;
    if (l < L)
      while (c < lim && stage[l * P + c] >= bound) ++c;
    int incl = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(kFullMask, incl, d);
      if (lane >= d) incl += y;
    }
    int at = 0;
    if (lane == 31 && incl > 0) at = atomicAdd(&s_count, incl);
    at = __shfl_sync(kFullMask, at, 31) + incl - c;
    for (int i = 0; i < c; ++i, ++at)
      if (at < kSurvivorCap) surv[at] = stage[l * P + i];
    unsigned more = __ballot_sync(kFullMask, l < L && c == lim && lim < k);
    while (more) {
      const int src = __ffs(more) - 1;
      more &= more - 1;
      const int lm = l0 + warp * 32 + src;
      for (int e0 = lim; e0 < k; e0 += 32) {
        const int e = e0 + lane;
        const uint64_t key = e < k ? list_key(p, base, lm, e) : 0ull;
        const bool pass = key >= bound;
        const unsigned msk = __ballot_sync(kFullMask, pass);
        if (msk == 0) break;
        int a = 0;
        if (lane == 0) a = atomicAdd(&s_count, __popc(msk));
        a = __shfl_sync(kFullMask, a, 0) + __popc(msk & ((1u << lane) - 1u));
        if (pass && a < kSurvivorCap) surv[a] = key;
        if (msk != kFullMask) break;
      }
    }
  }
  __syncthreads();
  const int S = s_count;
  if (S > kSurvivorCap) return false;
  if (tid == 0) {
    surv[S] = 0;  // pad to an even count for paired reads; 0 beats nothing
    surv[S + 1] = 0;
  }
  __syncthreads();
  const ulonglong2* pairs = reinterpret_cast<const ulonglong2*>(surv);
  for (int i = tid; i < S; i += NT) {
    const uint64_t x = surv[i];
    int place = 0;
    for (int j = 0; j < (S + 1) / 2; ++j) {
      const ulonglong2 g = pairs[j];
      place += (g.x > x ? 1 : 0) + (g.y > x ? 1 : 0);
    }
    if (place < k) emit(p, place, x);
  }
  for (int e = S + tid; e < k; e += NT) emit(p, e, 0ull);  // fewer than K real keys
  return true;
}


// The general merge: lists staged stage_lists at a time after WARPS lists of
// KP >= K keys used as the tree; each warp folds a strided subset of the staged
// lists into its register list, then the warp lists merge pairwise.
template <int KP, int NT>
__device__ void merge_general(const MergeOut& p, const uint64_t* base, int L, uint64_t* smem, int stage_lists) {
  constexpr int R = KP / 32;
  constexpr int WARPS = NT / 32;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint64_t* lists = smem;               // WARPS lists of KP keys (the tree)
  uint64_t* stage = smem + WARPS * KP;  // staged list heads, k keys each
  uint64_t v[R];
  warp_list_clear<R>(v);
  for (int g0 = 0; g0 < L; g0 += stage_lists) {
    const int gl = min(stage_lists, L - g0);
    stage_heads<NT>(p, stage, base, g0, gl, p.k);
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
    if ((warp % (2 * step)) == 0 && warp + step < WARPS) {
      warp_list_merge_from<R>(v, lists + (warp + step) * KP, lane);
      warp_list_store<R>(v, lists + warp * KP, lane);
    }
    __syncthreads();
  }
  if (warp == 0) {
#pragma unroll
    for (int s = 0; s < R; ++s) {
      const int e = s * 32 + lane;
      if (e < p.k) emit(p, e, v[s]);
    }
  }
}

// One query's merge by all NT threads of the CTA over the L lists at base
// (KP >= K: the register list width of the general merge), in smem_bytes of
// dynamic shared memory (at least fast_smem_bytes(L, k, stage_keys) or, for
// the general merge, room for NT/32 lists of KP keys and one staged list). Block-uniform; ends with the
// outputs written (no barrier after the last write).
template <int KP, int NT>
__device__ void merge_lists(const MergeOut& p, const uint64_t* base, int L, uint64_t* smem, int smem_bytes,
                            int stage_keys) {
  if (!merge_fast<KP, NT>(p, base, L, smem, stage_keys)) {
    __syncthreads();  // the fast path's shared memory is reused below
    const int room = smem_bytes / 8 - (NT / 32) * KP;
    const int stage_lists = max(1, min(L, room / p.k));
    merge_general<KP, NT>(p, base, L, smem, stage_lists);
  }
}

}  // namespace mergecore
}  // namespace rbf
