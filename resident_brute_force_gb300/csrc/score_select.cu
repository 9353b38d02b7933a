// score_select.cu -- fused inner-product scoring + per-CTA partial top-K.
//
// One pass over the resident corpus per query (GPU-Resident Top-K for Agentic
// RAG, section 4 steps 2 and 3: score every row, then each block keeps a
// best-first top-K of its rows). Here the two steps are one kernel and the N
// scores never leave the SM:
//
//   * persistent grid, one CTA per SM (or a few); each CTA takes tiles of
//     consecutive rows, either a static contiguous range or by claiming tiles
//     from a global counter;
//   * a producer warp streams tiles HBM -> shared memory with one-dimensional
//     bulk copies (TMA) into an S-stage ring guarded by full/empty mbarriers;
//   * eight consumer warps each take whole rows: every lane reads 16-byte
//     chunks of the row (a warp reads 512 contiguous bytes per instruction,
//     conflict-free), multiplies with the query held in registers, and a
//     butterfly shuffle reduction finishes the row. Every row is reduced in
//     the same order wherever it sits, so equal rows get bit-equal scores;
//   * each warp keeps its best KP keys in a register bitonic list with a
//     threshold (its K-th key); rows that beat it are buffered one per lane
//     and merged 32 at a time;
//   * at the end the CTA merges its warps' lists in shared memory and writes
//     one best-first list of KP keys;
//   * with output pointers, the last CTA to finish (a ticket after a fence)
//     then merges all the lists itself (section 4 step 4) in the ring's
//     shared memory and hands over the call's error word, so a search is one
//     launch; without them the lists are left for the merge kernel.
#include "merge_core.cuh"
#include "rbf_device.cuh"
#include "rbf_internal.h"

namespace rbf {
namespace {

constexpr int NW = kScoreConsumerWarps;
constexpr int kThreads = (NW + 1) * 32;

// Keys the fused merge may stage in a ring of `bytes` (the rest holds the
// survivors).
__host__ __device__ constexpr int merge_stage_keys(int bytes) {
  return (bytes / 8 - mergecore::kSurvivorCap - 2) & ~1;
}

struct Params {
  const float* corpus;
  const float* query;
  uint64_t* partials;
  int* err;
  unsigned* counters;
  int64_t n;
  int d;
  int pitch;
  int k;
  int rows_per_stage;
  int stages;
  int stage_bytes;
  int region_bytes;  // ring bytes, or the list scratch if larger
  int dynamic;
  uint64_t timeout_ns;
  // Merge in the last CTA (when out_idx is set): K indices and scores, and
  // the per-call error word handed to result_err / err_sticky.
  int32_t* out_idx;
  float* out_score;
  int* err_sticky;
  int* result_err;
  size_t partials_cap;  // keys (checked builds; 0: not checked)
  uint32_t index_offset;  // added to every row index (global rows of a shard)
  int host_result;        // 1: results in mapped host memory, the host waits on result_err
};

// NCH > 0: rows are exactly NCH * 128 floats and the query lives in
// registers. NCH == 0: any pitch, query read from shared memory. NORM:
// cosine mode, the kernel first scales its copy of the query to unit length.
template <int KP, int NCH, bool NORM>
__global__ void __launch_bounds__(kThreads, 1) score_select_f32_kernel(const Params p) {
  constexpr int R = KP / 32;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.region_bytes);
  uint64_t* empty = full + p.stages;
  int64_t* hdr_row0 = reinterpret_cast<int64_t*>(empty + p.stages);
  int* hdr_rows = reinterpret_cast<int*>(hdr_row0 + p.stages);
  float* sq = reinterpret_cast<float*>(smem + p.region_bytes + p.stages * 32);
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int RS = p.rows_per_stage;
  const int64_t total_tiles = (p.n + RS - 1) / RS;
  // With dynamic claims CTA b's first tile is tile b, issued before the wait
  // on the previous kernel below: the corpus is never written by a kernel
  // (an upload synchronises the stream), so the copy may overlap that
  // kernel's tail. The claims then start at tile gridDim.x.
  const bool first_early = p.dynamic && blockIdx.x < total_tiles;
  pdl_launch_dependents();  // the merge kernel may be scheduled now; it waits for us

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NW);
    }
    fence_mbar_init();
    if (first_early) {
      const int64_t row0 = static_cast<int64_t>(blockIdx.x) * RS;
      const int rows = static_cast<int>(min(p.n, row0 + RS) - row0);
      const uint32_t bytes = static_cast<uint32_t>(rows) * static_cast<uint32_t>(p.pitch) * 4u;
      hdr_row0[0] = row0;
      hdr_rows[0] = rows;
      mbar_arrive_expect_tx(&full[0], bytes);
      bulk_copy_g2s(ring, p.corpus + row0 * p.pitch, bytes, &full[0], l2_policy_evict_first());
    }
  }
  // Launched as a programmatic dependent of the previous kernel on the
  // stream: this CTA may become resident while that kernel's last CTA is
  // still merging. Nothing above touched global memory; everything below
  // (the query, the tile counters, the lists) waits for that kernel.
  pdl_wait();
  if constexpr (NCH == 0) {
    for (int i = threadIdx.x; i < p.pitch; i += blockDim.x) sq[i] = (i < p.d) ? p.query[i] : 0.0f;
    if constexpr (NORM) {
      // Cosine mode: the shared copy scaled to unit length (fp32 sum of
      // squares in a fixed order, so every CTA gets the same bits).
      __shared__ float s_part[NW + 1];
      __shared__ float s_inv;
      __syncthreads();
      float ss = 0.0f;
      for (int i = threadIdx.x; i < p.d; i += blockDim.x) ss = fmaf(sq[i], sq[i], ss);
#pragma unroll
      for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(kFullMask, ss, m);
      if (lane == 0) s_part[warp] = ss;
      __syncthreads();
      if (threadIdx.x == 0) {
        float t = 0.0f;
        for (int w = 0; w <= NW; ++w) t += s_part[w];
        s_inv = inv_l2_norm_f(t);
      }
      __syncthreads();
      for (int i = threadIdx.x; i < p.d; i += blockDim.x) sq[i] *= s_inv;
    }
  }
  __syncthreads();

  uint64_t v[R];
  warp_list_clear<R>(v);

  if (warp == NW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      const int64_t row_bytes = static_cast<int64_t>(p.pitch) * 4;
      const int64_t r0 = p.n * blockIdx.x / gridDim.x;
      const int64_t r1 = p.n * (blockIdx.x + 1) / gridDim.x;
      const int64_t local_tiles = (r1 - r0 + RS - 1) / RS;
      int64_t claim = p.dynamic ? static_cast<int64_t>(atomicAdd(&p.counters[0], 1u)) + gridDim.x : 0;
      int64_t issued = first_early ? 1 : 0;  // the first tile, issued in the prologue
      bool aborted = false;
      for (int64_t i = issued;; ++i) {
        const int s = static_cast<int>(i % p.stages);
        const uint32_t u = static_cast<uint32_t>(i / p.stages);
        const bool end = p.dynamic ? (claim >= total_tiles) : (i >= local_tiles);
        int64_t row0 = 0, row_end = 0;
        if (!end) {
          if (p.dynamic) {
            row0 = claim * RS;
            row_end = min(p.n, row0 + RS);
            claim = static_cast<int64_t>(atomicAdd(&p.counters[0], 1u)) + gridDim.x;  // next claim, in flight
          } else {
            row0 = r0 + i * RS;
            row_end = min(r1, row0 + RS);
          }
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
          // End marker: a header with no rows, completing the stage's phase
          // with a plain arrival (no bytes expected).
          hdr_rows[s] = -1;
          mbar_arrive(&full[s]);
          break;
        }
        const int rows = static_cast<int>(row_end - row0);
        const uint32_t bytes = static_cast<uint32_t>(rows * row_bytes);
        hdr_row0[s] = row0;
        hdr_rows[s] = rows;
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_copy_g2s(ring + static_cast<size_t>(s) * p.stage_bytes, p.corpus + row0 * p.pitch, bytes, &full[s],
                      pol);
        ++issued;
      }
      if (aborted) {
        // Something timed out. Before the CTA may exit, every copy still in
        // flight must land: the last `stages` issued tiles sit on distinct
        // stages and are the newest phase of each barrier, so their parity
        // waits are unambiguous. (On the normal path the consumers have
        // already waited on every issued tile.)
        abort_flag = 1;
        for (int64_t i = (issued > p.stages ? issued - p.stages : 0); i < issued; ++i) {
          const int s = static_cast<int>(i % p.stages);
          const uint32_t u = static_cast<uint32_t>(i / p.stages);
          if (!mbar_wait(&full[s], u & 1u, p.timeout_ns)) atomicOr(p.err, kErrDrainTimeout);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers
    float4 q[NCH > 0 ? NCH : 1];
    if constexpr (NCH > 0) {
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const int e = (lane + 32 * j) * 4;
        q[j].x = (e + 0 < p.d) ? p.query[e + 0] : 0.0f;
        q[j].y = (e + 1 < p.d) ? p.query[e + 1] : 0.0f;
        q[j].z = (e + 2 < p.d) ? p.query[e + 2] : 0.0f;
        q[j].w = (e + 3 < p.d) ? p.query[e + 3] : 0.0f;
      }
      if constexpr (NORM) {
        // Cosine mode: every consumer warp scales its register copy to unit
        // length (fp32 sum of squares, the same order in every warp).
        float ss = 0.0f;
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          ss = fmaf(q[j].x, q[j].x, ss);
          ss = fmaf(q[j].y, q[j].y, ss);
          ss = fmaf(q[j].z, q[j].z, ss);
          ss = fmaf(q[j].w, q[j].w, ss);
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(kFullMask, ss, m);
        const float inv = inv_l2_norm_f(ss);
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          q[j].x *= inv;
          q[j].y *= inv;
          q[j].z *= inv;
          q[j].w *= inv;
        }
      }
    }
    const float4* sq4 = reinterpret_cast<const float4*>(sq);
    const int pitch4 = p.pitch >> 2;
    uint64_t theta = 0;  // key of the warp's K-th best so far (0: list not full)
    uint64_t cand = 0;
    int cnt = 0;
    for (int64_t i = 0;; ++i) {
      const int s = static_cast<int>(i % p.stages);
      const uint32_t u = static_cast<uint32_t>(i / p.stages);
      // Every lane polls; the verdict is made warp-uniform so a timeout can
      // never split the warp ahead of the full-mask shuffles below.
      if (!__all_sync(kFullMask, mbar_wait(&full[s], u & 1u, p.timeout_ns))) {
        if (lane == 0) atomicOr(p.err, kErrConsumerTimeout);
        abort_flag = 1;
        break;
      }
      const int rows = hdr_rows[s];
      if (rows < 0 || *reinterpret_cast<volatile int*>(&abort_flag)) break;
      const int64_t row0 = hdr_row0[s];
      const float* base = reinterpret_cast<const float*>(ring + static_cast<size_t>(s) * p.stage_bytes);
      for (int r = warp; r < rows; r += NW) {
        const float4* row = reinterpret_cast<const float4*>(base + static_cast<size_t>(r) * p.pitch);
        float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
        if constexpr (NCH > 0) {
#pragma unroll
          for (int j = 0; j < NCH; ++j) {
            const float4 c = row[lane + 32 * j];
            a0 = fmaf(c.x, q[j].x, a0);
            a1 = fmaf(c.y, q[j].y, a1);
            a2 = fmaf(c.z, q[j].z, a2);
            a3 = fmaf(c.w, q[j].w, a3);
          }
        } else {
          for (int j = lane; j < pitch4; j += 32) {
            const float4 c = row[j];
            const float4 w = sq4[j];
            a0 = fmaf(c.x, w.x, a0);
            a1 = fmaf(c.y, w.y, a1);
            a2 = fmaf(c.z, w.z, a2);
            a3 = fmaf(c.w, w.w, a3);
          }
        }
        float acc = (a0 + a1) + (a2 + a3);
        acc += __shfl_xor_sync(kFullMask, acc, 16);
        acc += __shfl_xor_sync(kFullMask, acc, 8);
        acc += __shfl_xor_sync(kFullMask, acc, 4);
        acc += __shfl_xor_sync(kFullMask, acc, 2);
        acc += __shfl_xor_sync(kFullMask, acc, 1);
        const uint64_t key = make_key(acc, static_cast<uint32_t>(row0 + r) + p.index_offset);
        if (key > theta) {  // warp-uniform: every lane holds the same acc
          if (lane == cnt) cand = key;
          if (++cnt == 32) {
            warp_list_insert32<R>(v, cand, lane);
            theta = warp_list_get<R>(v, p.k - 1);
            cnt = 0;
            cand = 0;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (cnt > 0) warp_list_insert32<R>(v, cand, lane);
  }

  // ---------------------------------------------------------------- CTA merge
  __syncthreads();
  uint64_t* lists = reinterpret_cast<uint64_t*>(smem);  // reuses the ring
  if (warp < NW) warp_list_store<R>(v, lists + warp * KP, lane);
  __syncthreads();
#pragma unroll
  for (int step = 1; step < NW; step <<= 1) {
    if (warp < NW && (warp % (2 * step)) == 0 && warp + step < NW) {
      warp_list_merge_from<R>(v, lists + (warp + step) * KP, lane);
      warp_list_store<R>(v, lists + warp * KP, lane);
    }
    __syncthreads();
  }
  if (warp == 0 &&
      in_bounds(p.partials_cap == 0 || (static_cast<size_t>(blockIdx.x) + 1) * KP <= p.partials_cap, p.err))
    warp_list_store<R>(v, p.partials + static_cast<size_t>(blockIdx.x) * KP, lane);

  if (!p.dynamic && !p.out_idx) return;
  // The last CTA to finish re-arms the tile counter for the next launch and,
  // when asked, merges every CTA's list.
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
  if (s_last && p.out_idx) {
    __threadfence();
    mergecore::MergeOut o;
    o.k = p.k;
    o.int_keys = 0;
    o.out_a = p.out_idx;
    o.out_b = p.out_score;
    o.kth_out = nullptr;
    o.q = 0;
    o.stride = KP;
    o.lens = nullptr;
    o.region = static_cast<size_t>(gridDim.x) * KP;
    o.err = p.err;
    // The ring only (the barriers after it are left alone).
    mergecore::merge_lists<KP, kThreads>(o, p.partials, static_cast<int>(gridDim.x), reinterpret_cast<uint64_t*>(smem),
                                         p.region_bytes, merge_stage_keys(p.region_bytes));
    // Hand the per-call error word to the sticky word and re-arm it for the
    // next call, then publish it to the result block after the results.
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

template <int KP, int NCH, bool NORM>
cudaError_t launch_t(const Params& p, int grid, int smem, cudaStream_t stream) {
  auto fn = score_select_f32_kernel<KP, NCH, NORM>;
  // The launch size depends on the engine's options (at most the device's
  // opt-in limit less the kernel's static shared memory), so the limit is
  // raised to that maximum, once per device.
  static PerDeviceOnce once;
  const cudaError_t limit = once.run([fn] {
    cudaFuncAttributes fa;
    const cudaError_t e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                max_dynamic_smem() - static_cast<int>(fa.sharedSizeBytes));
  });
  if (limit != cudaSuccess) return limit;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, p);
}

template <int KP, bool NORM>
cudaError_t launch_kpn(const Params& p, int grid, int smem, cudaStream_t stream) {
  switch (p.pitch) {
    case 384: return launch_t<KP, 3, NORM>(p, grid, smem, stream);
    case 768: return launch_t<KP, 6, NORM>(p, grid, smem, stream);
    case 1024: return launch_t<KP, 8, NORM>(p, grid, smem, stream);
    default: return launch_t<KP, 0, NORM>(p, grid, smem, stream);
  }
}

template <int KP>
cudaError_t launch_kp(const Params& p, int grid, int smem, bool norm, cudaStream_t stream) {
  return norm ? launch_kpn<KP, true>(p, grid, smem, stream) : launch_kpn<KP, false>(p, grid, smem, stream);
}

int region_bytes(int pitch, int k, int rows_per_stage, int stages) {
  const int ring = stages * rows_per_stage * pitch * 4;
  const int lists = NW * list_width(k) * 8;
  return ring > lists ? ring : lists;
}

}  // namespace

bool score_select_can_merge(int pitch, int k, int rows_per_stage, int stages) {
  // The general merge needs a tree of one list per warp plus one staged
  // list; the fast path applies when its staging fits as well.
  const int keys = region_bytes(pitch, k, rows_per_stage, stages) / 8;
  return keys >= (kThreads / 32) * list_width(k) + k;
}

int score_select_smem_bytes(int pitch, int k, int rows_per_stage, int stages) {
  // region | full[S] empty[S] row0[S] rows[S] (32 B per stage) | query copy
  return region_bytes(pitch, k, rows_per_stage, stages) + stages * 32 + pitch * 4;
}

cudaError_t launch_score_select(const ScoreSelectLaunch& a, cudaStream_t stream) {
  Params p;
  p.corpus = a.corpus;
  p.query = a.query;
  p.partials = a.partials;
  p.err = a.err;
  p.counters = a.counters;
  p.n = a.n;
  p.d = a.d;
  p.pitch = a.pitch;
  p.k = a.k;
  p.rows_per_stage = a.rows_per_stage;
  p.stages = a.stages;
  p.stage_bytes = a.rows_per_stage * a.pitch * 4;
  p.region_bytes = region_bytes(a.pitch, a.k, a.rows_per_stage, a.stages);
  p.dynamic = a.dynamic;
  p.timeout_ns = a.timeout_ns;
  p.out_idx = a.out_idx;
  p.out_score = a.out_score;
  p.err_sticky = a.err_sticky;
  p.result_err = a.result_err;
  p.partials_cap = a.partials_cap;
  p.index_offset = a.index_offset;
  p.host_result = a.host_result;
  const int smem = score_select_smem_bytes(a.pitch, a.k, a.rows_per_stage, a.stages);
  switch (list_width(a.k)) {
    case 32: return launch_kp<32>(p, a.grid, smem, a.normalize_query != 0, stream);
    case 64: return launch_kp<64>(p, a.grid, smem, a.normalize_query != 0, stream);
    case 128: return launch_kp<128>(p, a.grid, smem, a.normalize_query != 0, stream);
    case 256: return launch_kp<256>(p, a.grid, smem, a.normalize_query != 0, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace rbf
