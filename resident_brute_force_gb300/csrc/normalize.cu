// normalize.cu -- cosine mode: unit-length rows and queries.
//
// Cosine similarity is the inner product divided by the product of the L2
// norms of the query and the row, and a row whose denominator is not
// positive scores -infinity (GPU-Resident Top-K for Agentic RAG, section 4
// step 2, the scoring kernel's cosine mode). The same article notes that
// dividing every row by its norm once at ingest turns cosine into a plain
// inner product. That is done here for the rows (at upload) and for the
// batched queries (at every call); the single-query scoring kernel scales its
// own copy of the query the same way. Norms are square roots of double sums of squares and
// every element is scaled in double, then rounded to fp32 once. A vector with
// zero norm (or a NaN or infinite element) becomes all NaN; its scores are
// NaN, which the selection keys rank as -infinity, as the rule asks.
#include <cuda_bf16.h>

#include <algorithm>

#include "rbf_device.cuh"
#include "rbf_internal.h"

namespace rbf {
namespace {

// Sum of squares of x[0..d) in double: lane-strided, then a fixed butterfly,
// so equal vectors give bit-equal norms.
__device__ __forceinline__ double warp_sumsq(const float* x, int d, int lane) {
  double ss = 0.0;
  for (int j = lane; j < d; j += 32) {
    const double v = static_cast<double>(x[j]);
    ss += v * v;
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(kFullMask, ss, m);
  return ss;
}

// One warp per row, in place: row[j] <- row[j] / ||row|| for j < d (the
// zero padding up to the pitch stays zero).
__global__ void normalize_rows_kernel(float* corpus, int64_t n, int d, int pitch) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); r < n; r += warps) {
    float* row = corpus + r * pitch;
    const double inv = inv_l2_norm(warp_sumsq(row, d, lane));
    for (int j = lane; j < d; j += 32) row[j] = static_cast<float>(static_cast<double>(row[j]) * inv);
  }
}

// One warp per query row: unit length, then bf16 (round to nearest even) into
// [rows_total][dst_pitch]; zero past `cols` and for rows in [rows, rows_total).
__global__ void normalize_queries_bf16_kernel(const float* __restrict__ src, int64_t src_pitch,
                                              __nv_bfloat16* __restrict__ dst, int64_t dst_pitch, int64_t rows,
                                              int64_t rows_total, int cols) {
  pdl_launch_dependents();  // the scoring pass may become resident now; its producer waits for these queries
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); r < rows_total;
       r += warps) {
    __nv_bfloat16* o = dst + r * dst_pitch;
    if (r < rows) {
      const float* x = src + r * src_pitch;
      const double inv = inv_l2_norm(warp_sumsq(x, cols, lane));
      for (int64_t j = lane; j < dst_pitch; j += 32)
        o[j] = __float2bfloat16_rn(j < cols ? static_cast<float>(static_cast<double>(x[j]) * inv) : 0.0f);
    } else {
      for (int64_t j = lane; j < dst_pitch; j += 32) o[j] = __float2bfloat16_rn(0.0f);
    }
  }
}

// fp32 queries into a padded fp32 buffer for the tf32 batched path: one warp
// per row, zero past `cols` and for rows in [rows, rows_total); with NORM the
// row is scaled to unit length first (cosine mode).
template <bool NORM>
__global__ void stage_queries_f32_kernel(const float* __restrict__ src, int64_t src_pitch, float* __restrict__ dst,
                                         int64_t dst_pitch, int64_t rows, int64_t rows_total, int cols) {
  pdl_launch_dependents();  // the scoring pass may become resident now; its producer waits for these queries
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); r < rows_total;
       r += warps) {
    float* o = dst + r * dst_pitch;
    if (r < rows) {
      const float* x = src + r * src_pitch;
      double inv = 1.0;
      if constexpr (NORM) inv = inv_l2_norm(warp_sumsq(x, cols, lane));
      for (int64_t j = lane; j < dst_pitch; j += 32) {
        if constexpr (NORM)
          o[j] = j < cols ? static_cast<float>(static_cast<double>(x[j]) * inv) : 0.0f;
        else
          o[j] = j < cols ? x[j] : 0.0f;
      }
    } else {
      for (int64_t j = lane; j < dst_pitch; j += 32) o[j] = 0.0f;
    }
  }
}

}  // namespace

cudaError_t launch_stage_queries_f32(const float* src, int64_t src_pitch, float* dst, int64_t dst_pitch, int64_t rows,
                                     int64_t rows_total, int cols, bool normalize, int num_sms, cudaStream_t st) {
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((rows_total + 7) / 8, int64_t(num_sms) * 4));
  if (normalize)
    stage_queries_f32_kernel<true><<<static_cast<int>(blocks), 256, 0, st>>>(src, src_pitch, dst, dst_pitch, rows,
                                                                           rows_total, cols);
  else
    stage_queries_f32_kernel<false><<<static_cast<int>(blocks), 256, 0, st>>>(src, src_pitch, dst, dst_pitch, rows,
                                                                            rows_total, cols);
  return cudaGetLastError();
}

cudaError_t launch_normalize_rows(float* corpus, int64_t n, int d, int pitch, int num_sms, cudaStream_t st) {
  const int64_t blocks = std::min<int64_t>((n + 7) / 8, int64_t(num_sms) * 16);
  normalize_rows_kernel<<<static_cast<int>(std::max<int64_t>(blocks, 1)), 256, 0, st>>>(corpus, n, d, pitch);
  return cudaGetLastError();
}

cudaError_t launch_normalize_queries_bf16(const float* src, int64_t src_pitch, void* dst, int64_t dst_pitch,
                                          int64_t rows, int64_t rows_total, int cols, int num_sms, cudaStream_t st) {
  const int64_t blocks = std::min<int64_t>((rows_total + 7) / 8, int64_t(num_sms) * 4);
  normalize_queries_bf16_kernel<<<static_cast<int>(std::max<int64_t>(blocks, 1)), 256, 0, st>>>(
      src, src_pitch, static_cast<__nv_bfloat16*>(dst), dst_pitch, rows, rows_total, cols);
  return cudaGetLastError();
}

}  // namespace rbf
