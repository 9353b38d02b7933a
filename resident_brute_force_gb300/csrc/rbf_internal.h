// rbf_internal.h -- host-side launch interfaces between the library's
// translation units. Not part of the public ABI (that is include/rbf.h).
#pragma once

#include <atomic>
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

namespace rbf {

// Consumer warps of the fused scoring kernel (plus one producer warp).
constexpr int kScoreConsumerWarps = 8;
// Warps of the int32 stage-1 kernel.
constexpr int kI32Warps = 16;

// The current device's opt-in dynamic shared-memory limit per block.
inline int max_dynamic_smem() {
  int dev = 0, bytes = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&bytes, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  return bytes;
}

// Runs a set-up step once per device, with that device current. A kernel's
// function attributes (its dynamic shared-memory limit) belong to the device
// that was current when they were set, so a process that launches on several
// devices must set them on each. One instance per kernel instance, kept as a
// function-local static at the launch site; after the first call on a device
// the cost is a cudaGetDevice and an atomic load.
class PerDeviceOnce {
 public:
  template <typename F>
  cudaError_t run(F&& setup) {
    int dev = 0;
    cudaError_t st = cudaGetDevice(&dev);
    if (st != cudaSuccess) return st;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (done_[dev].load(std::memory_order_acquire)) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    st = setup();
    if (st == cudaSuccess) done_[dev].store(true, std::memory_order_release);
    return st;
  }

 private:
  static constexpr int kMaxDevices = 64;
  std::atomic<bool> done_[kMaxDevices] = {};
  std::mutex mu_;
};

// Candidate-list width for a K: the smallest power of two >= max(K, 32).
inline int list_width(int k) {
  int kp = 32;
  while (kp < k) kp <<= 1;
  return kp;
}

struct ScoreSelectLaunch {
  const float* corpus;     // device, n rows of `pitch` floats, zero-padded past d
  const float* query;      // device, d floats
  uint64_t* partials;      // device, grid lists of list_width(k) keys
  int* err;                // device error word (bits ORed in)
  unsigned* counters;      // device, 2 words, zero between launches (dynamic schedule)
  int64_t n;
  int d;
  int pitch;               // floats per stored row, multiple of 4
  int k;
  int rows_per_stage;
  int stages;
  int stage_bytes;
  int grid;
  int dynamic;             // 0 = static contiguous row ranges, 1 = tile claims
  uint64_t timeout_ns;
  int normalize_query = 0; // 1: score with the query scaled to unit length (cosine mode)
  uint32_t index_offset = 0;  // added to every row index (a row shard's first global row)
  // Set: the last CTA merges the lists into K indices / scores (device or
  // mapped host memory) and hands the error word to result_err / err_sticky.
  int32_t* out_idx = nullptr;
  float* out_score = nullptr;
  int* err_sticky = nullptr;
  int* result_err = nullptr;
  int host_result = 0;      // 1: results in mapped host memory, the host waits on result_err
  size_t partials_cap = 0;  // keys in partials, for checked builds (0: not checked)
};

// Shared memory the fused kernel needs for a launch shape.
int score_select_smem_bytes(int pitch, int k, int rows_per_stage, int stages);
// Whether the kernel's ring can hold its last CTA's merge for this shape.
bool score_select_can_merge(int pitch, int k, int rows_per_stage, int stages);
cudaError_t launch_score_select(const ScoreSelectLaunch& a, cudaStream_t stream);

struct MergeLaunch {
  const uint64_t* partials;  // device, queries x lists x stride keys
  int lists;                 // lists per query
  int queries;               // one CTA per query
  int k;
  int int_keys;              // 0: (fp32 score, int32 index) keys; 1: (int32 value, position) keys
  int32_t* out_a;            // float path: indices [queries x k]; int path: values [k]
  void* out_b;               // float path: float scores; int path: int64 positions
  int* err_call;             // per-call error word, moved out and cleared
  int* err_sticky;           // sticky error word (ORed)
  int* result_err;           // where the per-call error lands (may be null)
  int host_result = 0;       // 1: one query, results in mapped host memory, the host waits on result_err
  uint64_t* kth_out = nullptr;  // optional: each query's K-th key
  int stride = 0;               // keys from one list to the next (0: list_width(k))
  const int* lens = nullptr;    // optional [queries x lists] valid keys per list (else all stride)
  size_t partials_cap = 0;      // keys in partials, for checked builds (0: not checked)
  int short_lists = 0;          // 1: lists hold few valid keys (K > 32): stage a 32-key prefix of each
};
cudaError_t launch_merge(const MergeLaunch& a, cudaStream_t stream);

// For each of `queries` queries, a lower bound on the K-th largest of its
// `total` keys (stored contiguously per query; keys of distinct rows, zero for
// none) into kth_out[query]: c << 32, c the largest score code that K of the
// keys reach; 0 if fewer than K are nonzero. total <= 1024, K <= 256.
constexpr int RBF_KTH_MAX_KEYS = 1024;
constexpr int RBF_KTH_MAX_K = 256;
cudaError_t launch_kth_of_lists(const uint64_t* keys, int queries, int total, int k, uint64_t* kth_out,
                                cudaStream_t stream);

// Row-sharded search: the best-first (index, score) lists of g shards for b
// queries, laid out [g][b][k] (index < 0: no entry), become keys in
// out[b][g][kp] (kp >= k; slots past k and missing entries hold the empty
// key), ready for launch_merge with g lists per query and stride kp.
cudaError_t launch_encode_shard_lists(const int32_t* idx, const float* score, int g, int b, int k, int kp,
                                      uint64_t* out, int num_sms, cudaStream_t stream);

struct I32Launch {
  const int32_t* data;
  int64_t n;
  int k;
  uint64_t* partials;        // grid lists of list_width(k) keys
  int grid;
  const uint64_t* theta0 = nullptr;  // optional lower bound on the K-th key (keys >= it are kept)
  size_t partials_cap = 0;           // keys in partials, for checked builds (0: not checked)
  int* err = nullptr;                // error word for checked builds (may be null)
};
cudaError_t launch_topk_i32_stage1(const I32Launch& a, cudaStream_t stream);

// Stage 1 for large arrays: bulk-copy ring, dynamic 64 KB tile claims, one
// CTA of 16 consumer warps + 1 producer per SM; each CTA bounds the K-th key
// from its own 32,768-value slice before its first tile. K <= 256.
struct I32StreamLaunch {
  const int32_t* data;
  int64_t n;
  int k;
  uint64_t* partials;          // grid lists of list_width(k) keys
  const uint64_t* theta0;      // optional lower bound on the K-th key (keys >= it are kept)
  unsigned* counters;          // 2 words, zero between launches
  int* err;                    // per-call error word
  int grid;
  uint64_t timeout_ns;
  // Optional stage 2 in the kernel's last CTA: K values and positions, and
  // the per-call error word handed to result_err / err_sticky (then cleared).
  int32_t* out_val = nullptr;
  int64_t* out_pos = nullptr;
  int* err_sticky = nullptr;
  int* result_err = nullptr;
  int host_result = 0;         // 1: results in mapped host memory, the host waits on result_err
  size_t partials_cap = 0;     // keys in partials, for checked builds (0: not checked)
};
cudaError_t launch_topk_i32_stream(const I32StreamLaunch& a, cudaStream_t stream);

cudaError_t launch_wait_probe(int* err, uint64_t timeout_ns, cudaStream_t stream);

// Cosine mode: unit-length rows (in place, at upload) and unit-length bf16
// queries for the batched path. A zero-norm vector becomes all NaN (scores
// -inf).
cudaError_t launch_normalize_rows(float* corpus, int64_t n, int d, int pitch, int num_sms, cudaStream_t st);
cudaError_t launch_normalize_queries_bf16(const float* src, int64_t src_pitch, void* dst, int64_t dst_pitch,
                                          int64_t rows, int64_t rows_total, int cols, int num_sms, cudaStream_t st);

// Batched queries (tensor cores). K <= 32; each launch covers up to 256
// queries; every CTA writes 32 keys per query.
constexpr int kBatchRegMaxK = 32;  // batched K up to this: per-thread lists in registers
constexpr int kBatchQueriesPerLaunch = 256;
constexpr int kBatchListWidth = 32;
constexpr int kBoundListWidth = 4;  // bound pre-pass: 4 chunk maxima per (query, CTA, column half)
constexpr int kBf16PitchAlign = 64;  // bf16 elements: one 128-byte swizzle row

struct GemmSelectLaunch {
  const void* tmap_q;        // host CUtensorMap over the bf16 query buffer
  const void* tmap_c;        // host CUtensorMap over the bf16 corpus
  uint64_t* partials;        // [queries][grid / 2][32] keys (one list per CTA pair); K > 32:
                             // [queries][grid][list_width(K)]; bound mode: [queries][grid][4]
  int* err;
  int64_t n;                 // corpus rows
  int kchunks;               // 128-byte K chunks per row (64 bf16 or 32 fp32 elements each)
  int tf32 = 0;              // 1: fp32 operands, kind::tf32 (tmap_c over the row-major fp32 corpus)
  int q_row0;                // first query row of this launch in the query buffer
  int q_count;               // queries in this launch, 1..256
  int q_out0;                // first query of this launch in the partials layout
  int k;
  int grid;                  // even: 2 x min(ceil(n / 256), SMs / 2)
  uint64_t timeout_ns;
  const uint64_t* theta0;    // optional per-query lower bound on the K-th key (keys >= it are kept)
  int bound_mode = 0;        // 1: no selection; each list (query, CTA, column half) holds the best key
                             // of each of 4 chunks of its rows (chunk c: columns 32c..32c+31 of its
                             // half of each tile), best first: kBoundListWidth keys per list
  int* lens = nullptr;       // K > 32: [queries][grid] valid keys of each list (required)
  int wait_inputs = 1;       // 1: the kernel launched just before wrote the queries (the producer waits
                             // for it); 0: the corpus stream may start while that kernel finishes
  size_t partials_cap = 0;   // keys in partials, lens entries, theta0 entries: for checked builds
  size_t lens_cap = 0;       // (0: not checked)
  size_t theta_cap = 0;
  uint32_t index_offset = 0; // added to every row index (a row shard's first global row)
};
// Tensor map over a [rows][pitch] bf16 matrix: 64 x 128 boxes, 128-byte swizzle.
bool make_bf16_tensor_map(void* map, const void* base, int64_t rows, int pitch_elems);
// Tensor map over a [rows][pitch] fp32 matrix: 32 x 128 boxes, 128-byte swizzle
// (the tf32 batched path: the resident corpus and the padded queries).
bool make_f32_tensor_map(void* map, const void* base, int64_t rows, int pitch_elems);
// fp32 queries [rows][src_pitch] -> [rows_total][dst_pitch] fp32, zero-padded,
// optionally scaled to unit length (cosine mode).
cudaError_t launch_stage_queries_f32(const float* src, int64_t src_pitch, float* dst, int64_t dst_pitch, int64_t rows,
                                     int64_t rows_total, int cols, bool normalize, int num_sms, cudaStream_t st);
// Corpus copy for the batched path, tile-major: [ceil(rows/128)][pitch/64][128][64]
// bf16, rows past `rows` zero. The map's box is one 16 KB block.
bool make_bf16_tiled_tensor_map(void* map, const void* base, int64_t rows, int pitch_elems);
cudaError_t launch_to_bf16_tiled(const float* src, int64_t src_pitch, void* dst, int64_t rows, int pitch_elems,
                                 int cols, int num_sms, cudaStream_t st);
cudaError_t launch_gemm_select(const GemmSelectLaunch& a, cudaStream_t stream);
// fp32 [rows][src_pitch] -> bf16 [rows_total][dst_pitch] (RN-even), zero padded.
cudaError_t launch_to_bf16(const float* src, int64_t src_pitch, void* dst, int64_t dst_pitch, int64_t rows,
                           int64_t rows_total, int cols, int num_sms, cudaStream_t stream);

}  // namespace rbf
