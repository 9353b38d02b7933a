// rbf_device.cuh -- device primitives shared by the sm_103a kernels.
//
//  * 64-bit selection keys that encode the ordering rule of GPU-Resident
//    Top-K for Agentic RAG (section 3, problem B: higher score first, lower
//    row index first on an exact tie) so that one unsigned compare decides
//    "better".
//  * mbarrier + bulk-copy (TMA) wrappers in inline PTX, with every wait
//    bounded by a time limit.
//  * Warp-wide sorted candidate lists kept in registers and merged with
//    bitonic networks (shuffles across lanes, register swaps across slots).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace rbf {

constexpr unsigned kFullMask = 0xFFFFFFFFu;

// Device error bits, ORed into the engine's error word.
constexpr int kErrConsumerTimeout = 1;
constexpr int kErrProducerTimeout = 2;
constexpr int kErrDrainTimeout = 4;
constexpr int kErrProbeTimeout = 8;
constexpr int kErrBounds = 16;  // a checked build met an index outside its buffer

// Checked builds (-DRBF_CHECKS): true when the access may go ahead; else the
// bounds bit is ORed into the error word and the caller skips the access.
// Other builds compile the check away. Used on the indices the kernels derive
// (list slots, list lengths, per-query offsets), not on the bulk and tensor
// copies, whose extents come straight from N and the tile sizes.
#ifdef RBF_CHECKS
__device__ __forceinline__ bool in_bounds(bool ok, int* err) {
  if (!ok && err) atomicOr(err, kErrBounds);
  return ok;
}
#else
__device__ __forceinline__ bool in_bounds(bool, int*) { return true; }
#endif

// The error word of a call whose results go to the host is written last,
// over this mark that the host left there before the launch: the host may
// wait for the word to change instead of synchronising the stream. Real
// error words are ORs of the kErr bits above.
constexpr int kResultPending = 0x40000000;

// Publish a one-CTA call's error word after its results. For results in
// host memory that the host waits on (host_result), every thread's writes
// reach system scope first; device-memory results need no fence (the stream
// orders them). Block-uniform.
__device__ __forceinline__ void publish_result_word(int* result_err, int e, bool host_result) {
  if (host_result) {
    __threadfence_system();
    __syncthreads();
    if (threadIdx.x == 0 && result_err) {
      __threadfence_system();
      *reinterpret_cast<volatile int*>(result_err) = e;
    }
  } else if (threadIdx.x == 0 && result_err) {
    *result_err = e;
  }
}

// ----------------------------------------------------------------- keys
//
// A key packs (score, index) so that key_a > key_b exactly when a is better
// than b under the ordering rule:
//   high 32 bits: the fp32 score mapped to an unsigned order-preserving code
//                 (NaN -> -inf, -0 -> +0 first),
//   low 32 bits:  0xFFFFFFFF - index (a lower index gives a larger key).
// The all-zero key is never produced by a real row (its score code would be a
// NaN pattern) and ranks below every real row: it is the empty-slot sentinel.

__device__ __forceinline__ uint32_t score_code(float s) {
  uint32_t b = __float_as_uint(s);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) b = 0xFF800000u;  // NaN -> -inf
  if (b == 0x80000000u) b = 0u;                          // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float score_from_code(uint32_t c) {
  const uint32_t b = (c & 0x80000000u) ? (c & 0x7FFFFFFFu) : ~c;
  return __uint_as_float(b);
}

__device__ __forceinline__ uint64_t make_key(float score, uint32_t index) {
  return (static_cast<uint64_t>(score_code(score)) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - index);
}

__device__ __forceinline__ uint32_t key_index(uint64_t key) {
  return 0xFFFFFFFFu - static_cast<uint32_t>(key);
}

__device__ __forceinline__ float key_score(uint64_t key) {
  return score_from_code(static_cast<uint32_t>(key >> 32));
}

// int32 values: order-preserving code is the sign-flipped pattern. Positions
// must stay below 2^32 - 1 so the sentinel stays unique.
__device__ __forceinline__ uint64_t make_ikey(int32_t value, uint32_t position) {
  return (static_cast<uint64_t>(static_cast<uint32_t>(value) ^ 0x80000000u) << 32) |
         static_cast<uint64_t>(0xFFFFFFFFu - position);
}

__device__ __forceinline__ int32_t ikey_value(uint64_t key) {
  return static_cast<int32_t>(static_cast<uint32_t>(key >> 32) ^ 0x80000000u);
}

__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }
__device__ __forceinline__ uint64_t umin64(uint64_t a, uint64_t b) { return a < b ? a : b; }

// 1 / sqrt(ss) for a sum of squares ss (cosine mode), or NaN when the norm is
// zero or not finite: such a vector then scores NaN everywhere, which the
// selection keys rank as -infinity.
__device__ __forceinline__ double inv_l2_norm(double ss) {
  return (ss > 0.0 && ss <= 1.7976931348623157e308) ? 1.0 / sqrt(ss) : __longlong_as_double(0x7FF8000000000000ll);
}
__device__ __forceinline__ float inv_l2_norm_f(float ss) {
  return (ss > 0.0f && ss <= 3.402823466e38f) ? 1.0f / sqrtf(ss) : __int_as_float(0x7FC00000);
}

// ------------------------------------------------------- timers, mbarriers

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait until the phase with the given parity has completed, or until
// timeout_ns has passed. Returns false on timeout. Every pipeline wait in the
// library goes through here, so no kernel can spin forever.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > timeout_ns) return false;
  }
}

// Programmatic dependent launch. A kernel launched with programmatic stream
// serialisation may start while the previous kernel on the stream is still
// running; pdl_wait() blocks until that kernel has finished and its writes are
// visible. pdl_launch_dependents() lets the next kernel be scheduled early.
// Both are no-ops when the launch carries no such dependency.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// L2 policy for data read exactly once per call: evict first.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// One-dimensional bulk copy global -> shared, completing `bytes` of
// transaction count on `bar`. dst and src 16-byte aligned, bytes a multiple
// of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// ------------------------------------------------------- warp key lists
//
// A warp list holds KP = 32 * R keys sorted in descending order (best
// first). Element e lives in lane (e % 32), register slot (e / 32).

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int m) { return __shfl_xor_sync(kFullMask, v, m); }
__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, int src) { return __shfl_sync(kFullMask, v, src); }

// Bitonic sort of one key per lane, descending across lanes (lane 0 best).
__device__ __forceinline__ uint64_t warp_sort32_desc(uint64_t v, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint64_t p = shfl_xor_u64(v, j);
      const bool lower = (lane & j) == 0;
      const bool desc = (lane & k) == 0;
      v = (lower == desc) ? umax64(v, p) : umin64(v, p);
    }
  }
  return v;
}

// Sort a bitonic sequence of KP = 32 * R keys into descending order
// (half-cleaner network: element strides KP/2 .. 1).
template <int R>
__device__ __forceinline__ void warp_bitonic_merge_desc(uint64_t (&v)[R], int lane) {
#pragma unroll
  for (int js = R / 2; js > 0; js >>= 1) {
#pragma unroll
    for (int s = 0; s < R; ++s) {
      if ((s & js) == 0) {
        const uint64_t a = v[s], b = v[s + js];
        v[s] = umax64(a, b);
        v[s + js] = umin64(a, b);
      }
    }
  }
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const bool lower = (lane & j) == 0;
#pragma unroll
    for (int s = 0; s < R; ++s) {
      const uint64_t p = shfl_xor_u64(v[s], j);
      v[s] = lower ? umax64(v[s], p) : umin64(v[s], p);
    }
  }
}

template <int R>
__device__ __forceinline__ void warp_list_clear(uint64_t (&v)[R]) {
#pragma unroll
  for (int s = 0; s < R; ++s) v[s] = 0;
}

// Merge 32 unsorted candidate keys (one per lane; 0 = empty) into the list,
// keeping the best KP of the union. The candidates are sorted, reversed and
// folded onto the last 32 elements with max(): the result is bitonic and holds
// the best KP of both, and a bitonic merge restores the order.
template <int R>
__device__ __forceinline__ void warp_list_insert32(uint64_t (&v)[R], uint64_t cand, int lane) {
  cand = warp_sort32_desc(cand, lane);
  const uint64_t rev = shfl_u64(cand, 31 - lane);
  v[R - 1] = umax64(v[R - 1], rev);
  warp_bitonic_merge_desc<R>(v, lane);
}

// Merge another descending list of KP keys, read from memory, into v.
template <int R>
__device__ __forceinline__ void warp_list_merge_from(uint64_t (&v)[R], const uint64_t* other, int lane) {
  constexpr int KP = 32 * R;
#pragma unroll
  for (int s = 0; s < R; ++s) v[s] = umax64(v[s], other[KP - 1 - (s * 32 + lane)]);
  warp_bitonic_merge_desc<R>(v, lane);
}

template <int R>
__device__ __forceinline__ void warp_list_store(const uint64_t (&v)[R], uint64_t* dst, int lane) {
#pragma unroll
  for (int s = 0; s < R; ++s) dst[s * 32 + lane] = v[s];
}

// Element e of the list, broadcast to every lane.
template <int R>
__device__ __forceinline__ uint64_t warp_list_get(const uint64_t (&v)[R], int e) {
  uint64_t x = 0;
  const int slot = e >> 5;
#pragma unroll
  for (int s = 0; s < R; ++s)
    if (s == slot) x = v[s];
  return shfl_u64(x, e & 31);
}

}  // namespace rbf
