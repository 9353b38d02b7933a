// engine.cu -- the engine behind the C ABI in include/rbf.h.
//
// The engine follows GPU-Resident Top-K for Agentic RAG (section 3 problem C
// and section 4 steps 0-6): every device buffer is allocated once, sized for
// the worst case, when the engine is created; the corpus is uploaded once and
// stays resident; each query then costs one small host-to-device copy, the
// kernels, and one small device-to-host copy of the K results. Here the
// per-query kernels are the fused score + partial select kernel and the merge
// kernel (score_select.cu, merge.cu); the flat int32 path is topk_i32.cu +
// merge.cu.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/rbf.h"
#include "rbf_device.cuh"
#include "rbf_internal.h"

using namespace rbf;

namespace {

constexpr int kMaxBatch = 4096;
constexpr int kResultHeader = 16;  // error word + padding, ahead of the results
constexpr int kMaxCtasPerSm = 4;
constexpr int kI32CtasPerSm = 2;
constexpr int64_t kSampleRows = 16384;  // rows of the batched path's threshold pre-pass
constexpr int64_t kI32StreamMin = 262144;   // int32 arrays at least this long take the stream kernel
constexpr int kI32SampleMinK = 65;          // from this K on, the stream kernel also gets a sample bound
constexpr int64_t kI32SampleElems = 65536;  // elements of that sample
constexpr int kMaxShards = 1024;            // lists one shard merge takes per query

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

struct rbf_engine {
  int device = 0;
  int num_sms = 0;
  int smem_optin = 0;
  cudaStream_t stream = nullptr;
  bool own_stream = false;

  int64_t max_n = 0;
  int max_d = 0, max_k = 0, max_batch = 0;
  uint32_t flags = 0;
  int max_pitch = 0;

  // Resident corpus.
  float* corpus = nullptr;
  int64_t n = 0;
  int d = 0;
  int pitch = 0;
  int64_t row_offset = 0;  // global index of the first resident row (row shards)
  bool ready = false;

  // bf16 copies for the batched path (RBF_FLAG_BF16_CORPUS).
  void* corpus_bf16 = nullptr;   // tile-major, max_n rounded up to 128 rows x max_pitch_bf16
  void* query_bf16 = nullptr;    // query_rows x max_pitch_bf16
  float* query_f32 = nullptr;    // tf32 batched path (no bf16 copy): query_rows x max_pitch floats
  uint64_t* theta0 = nullptr;    // per query: K-th key over the row sample
  int* lens = nullptr;           // batched K > 32: keys in each per-CTA list of a 256-query group
  int64_t batch_sample = -1;     // RBF_OPT_BATCH_SAMPLE
  int host_read = 0;             // RBF_OPT_HOST_READ: kernels may read the caller's pageable host buffers
  int host_read_ok = 0;          // the device reads pageable host memory through the host's page tables
  int max_pitch_bf16 = 0;
  int pitch_bf16 = 0;
  int query_rows = 0;            // max_batch rounded up to 256
  CUtensorMap tmap_corpus;  // the type carries the alignment a tensor map needs
  CUtensorMap tmap_query;
  bool tmaps_ready = false;

  // Workspaces (device).
  uint64_t* partials = nullptr;  // partials_cap keys
  uint64_t* i32_theta0 = nullptr;  // int32 path: K-th key of the element sample
  size_t partials_cap = 0;
  int* errw = nullptr;           // [0] per call, [1] sticky, [2] self-test
  unsigned* counters = nullptr;  // tile-claim counters: [0..1] scoring kernel, [2..3] int32 stream
  uint8_t* result = nullptr;     // device result block
  size_t result_bytes = 0;

  // Pinned host staging.
  uint8_t* h_query = nullptr;
  const float* d_hquery = nullptr;  // h_query as the device addresses it (pinned, mapped)
  uint8_t* h_result = nullptr;
  uint8_t* d_hres = nullptr;     // h_result as the device addresses it (pinned, mapped)
  // search_resident as one CUDA graph per K (query copy, scoring, merge),
  // captured on first use and dropped whenever the corpus or an option changes.
  cudaGraphExec_t host_graph[RBF_MAX_K + 1] = {};
  int host_graph_lists[RBF_MAX_K + 1] = {};
  int host_graph_launches[RBF_MAX_K + 1] = {};

  // Options.
  int ctas_per_sm = 1;
  int stage_bytes = 65536;
  int smem_budget = 0;  // 0: derived from the device limit
  uint64_t timeout_ns = 2000000000ull;
  int dynamic = 1;

  // Last scoring launch (for merge_partial_topk_dev).
  int last_lists = 0;
  int last_k = 0;

  int last_cuda_error = 0;
  int launches = 0;  // kernels enqueued by the most recent call (rbf_last_launches)
  int fault_kind = 0;
  int fault_count = 0;

  // Views (rbf_create_view): a view searches its owner's corpus with its own
  // stream and per-call buffers. The owner lists its views (an upload waits
  // for their streams) and bumps corpus_version around every upload; a view
  // re-reads the corpus state when the version it saw is stale.
  rbf_engine* owner = nullptr;
  std::vector<rbf_engine*> views;
  std::mutex views_mu;  // views may be made and destroyed from several host threads
  unsigned corpus_version = 0;
  unsigned seen_version = 0;
};

namespace {

rbf_status cuda_fail(rbf_engine* e, cudaError_t err) {
  if (e) e->last_cuda_error = static_cast<int>(err);
  return RBF_ERR_CUDA;
}

// Host-side fault injection: report a failure instead of issuing the next
// operation of the armed kind.
bool inject(rbf_engine* e, int kind) {
  if (e->fault_count > 0 && e->fault_kind == kind) {
    --e->fault_count;
    e->last_cuda_error = static_cast<int>(cudaErrorUnknown);
    return true;
  }
  return false;
}

// The partials capacity the kernels check their list slots against (checked
// builds). There RBF_FAULT=bounds understates it, so that the checks fire --
// the accesses are skipped and the bounds bit set -- without any access
// outside the buffer.
size_t device_cap(const rbf_engine* e) {
#ifdef RBF_CHECKS
  const char* v = std::getenv("RBF_FAULT");
  if (v && std::strcmp(v, "bounds") == 0) return 64;
#endif
  return e->partials_cap;
}

#define RBF_COPY(e, call)                              \
  do {                                                 \
    if (inject((e), 1)) return RBF_ERR_CUDA;           \
    cudaError_t _st = (call);                          \
    if (_st != cudaSuccess) return cuda_fail((e), _st); \
  } while (0)

#define RBF_LAUNCH(e, call)                            \
  do {                                                 \
    if (inject((e), 2)) return RBF_ERR_CUDA;           \
    cudaError_t _st = (call);                          \
    if (_st != cudaSuccess) return cuda_fail((e), _st); \
    ++(e)->launches;                                   \
  } while (0)

struct ScoreShape {
  int rows_per_stage = 0;
  int stages = 0;
  int grid = 0;
  int smem = 0;
};

// Launch shape of the fused scoring kernel for the resident corpus.
bool score_shape(const rbf_engine* e, int k, ScoreShape* out) {
  const int row_bytes = e->pitch * 4;
  int budget = e->smem_budget;
  if (budget <= 0) budget = std::min(e->smem_optin - 2048, 200 * 1024) / e->ctas_per_sm;
  const int fixed = e->pitch * 4;  // query copy
  for (int rps = std::max(1, e->stage_bytes / row_bytes); rps >= 1; rps = (rps > 1 ? rps / 2 : 0)) {
    const int sb = rps * row_bytes;
    int stages = (budget - fixed) / (sb + 32);
    stages = std::min(stages, 32);
    if (stages >= 2) {
      const int smem = score_select_smem_bytes(e->pitch, k, rps, stages);
      if (smem > e->smem_optin) continue;
      out->rows_per_stage = rps;
      out->stages = stages;
      const int64_t tiles = (e->n + rps - 1) / rps;
      out->grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(tiles, int64_t(e->num_sms) * e->ctas_per_sm)));
      out->smem = smem;
      return true;
    }
    if (rps == 1) break;
  }
  return false;
}

rbf_status check_k(const rbf_engine* e, int k) {
  if (k < 1 || k > e->max_k || k > RBF_MAX_K || static_cast<int64_t>(k) > e->n) return RBF_ERR_INVALID_VALUE;
  return RBF_OK;
}

// The scoring kernel over the resident corpus; with d_idx set its last CTA
// also merges the lists into the outputs (one launch per search), else the
// lists stay for enqueue_merge (last_lists). *merged tells which happened.
rbf_status enqueue_score(rbf_engine* e, const float* d_query, int k, int32_t* d_idx = nullptr,
                         float* d_score = nullptr, int* result_err = nullptr, bool* merged = nullptr,
                         bool host_result = false) {
  ScoreShape sh;
  if (!score_shape(e, k, &sh)) return RBF_ERR_UNSUPPORTED;
  if (static_cast<size_t>(sh.grid) * list_width(k) > e->partials_cap) return RBF_ERR_UNSUPPORTED;
  ScoreSelectLaunch a;
  a.corpus = e->corpus;
  a.query = d_query;
  a.partials = e->partials;
  a.err = e->errw;
  a.counters = e->counters;
  a.n = e->n;
  a.d = e->d;
  a.pitch = e->pitch;
  a.k = k;
  a.rows_per_stage = sh.rows_per_stage;
  a.stages = sh.stages;
  a.stage_bytes = sh.rows_per_stage * e->pitch * 4;
  a.grid = sh.grid;
  a.dynamic = e->dynamic;
  a.timeout_ns = e->timeout_ns;
  a.partials_cap = device_cap(e);
  // Cosine mode: rows are unit length already; the kernel scales its copy of
  // the query to unit length, so the inner product is the cosine.
  a.normalize_query = (e->flags & RBF_FLAG_COSINE) ? 1 : 0;
  a.index_offset = static_cast<uint32_t>(e->row_offset);
  const bool fuse = d_idx && score_select_can_merge(e->pitch, k, sh.rows_per_stage, sh.stages);
  if (fuse) {
    a.out_idx = d_idx;
    a.out_score = d_score;
    a.err_sticky = e->errw + 1;
    a.result_err = result_err;
    a.host_result = host_result ? 1 : 0;
  }
  RBF_LAUNCH(e, launch_score_select(a, e->stream));
  e->last_lists = sh.grid;
  e->last_k = k;
  if (merged) *merged = fuse;
  return RBF_OK;
}

rbf_status enqueue_merge(rbf_engine* e, int k, int lists, int queries, int int_keys, int32_t* out_a, void* out_b,
                         int* result_err, bool host_result = false) {
  MergeLaunch m;
  m.partials = e->partials;
  m.lists = lists;
  m.queries = queries;
  m.k = k;
  m.int_keys = int_keys;
  m.out_a = out_a;
  m.out_b = out_b;
  m.err_call = e->errw;
  m.err_sticky = e->errw + 1;
  m.result_err = result_err;
  m.host_result = host_result && queries == 1 ? 1 : 0;
  m.partials_cap = device_cap(e);
  RBF_LAUNCH(e, launch_merge(m, e->stream));
  return RBF_OK;
}

// Result block layout for `count` results: [err | pad][a: 4*count][b: eb*count]
struct ResultLayout {
  size_t a_off, b_off, bytes;
};

ResultLayout result_layout(size_t count, size_t eb) {
  ResultLayout r;
  r.a_off = kResultHeader;
  r.b_off = align_up(r.a_off + 4 * count, 16);
  r.bytes = r.b_off + eb * count;
  return r;
}

// The merge of a host-buffer call writes its results and the call's error
// word straight into the pinned host block (no separate device-to-host copy),
// so finishing the call is a stream synchronisation.
rbf_status finish_host_call(rbf_engine* e, const ResultLayout& L) {
  (void)L;
  cudaError_t st = cudaStreamSynchronize(e->stream);
  if (st != cudaSuccess) return cuda_fail(e, st);
  int derr = 0;
  std::memcpy(&derr, e->h_result, sizeof(int));
  if (derr & kErrBounds) return RBF_ERR_BOUNDS;
  if (derr != 0) return RBF_ERR_TIMEOUT;
  return RBF_OK;
}

// The error word of a one-CTA call's results (a single-query search, an
// int32 top-K) is written by the device after the results, over the
// kResultPending mark left here before the launch.
void mark_result_pending(rbf_engine* e) { reinterpret_cast<volatile int*>(e->h_result)[0] = kResultPending; }

// Wait for such a call by watching its error word in the pinned result block,
// which lands (over NVLink-C2C on GB300) as soon as the kernel writes it,
// sooner than a stream synchronisation returns; the stream is queried every
// 256 reads, so a launch that fails or finishes without writing the word
// ends the wait too. The results are in place when the word has changed.
rbf_status finish_host_call_polled(rbf_engine* e) {
  volatile int* w = reinterpret_cast<volatile int*>(e->h_result);
  for (unsigned spin = 1; *w == kResultPending; ++spin) {
    if ((spin & 255u) == 0) {
      const cudaError_t st = cudaStreamQuery(e->stream);
      if (st == cudaSuccess) break;
      if (st != cudaErrorNotReady) return cuda_fail(e, st);
    }
  }
  std::atomic_thread_fence(std::memory_order_acquire);
  const int derr = *w;
  if (derr == kResultPending) {  // the stream finished without the word: report it, don't read stale results
    const cudaError_t st = cudaStreamSynchronize(e->stream);
    return cuda_fail(e, st != cudaSuccess ? st : cudaErrorUnknown);
  }
  if (derr & kErrBounds) return RBF_ERR_BOUNDS;
  if (derr != 0) return RBF_ERR_TIMEOUT;
  return RBF_OK;
}

void drop_graphs(rbf_engine* e) {
  for (auto& g : e->host_graph) {
    if (g) cudaGraphExecDestroy(g);
    g = nullptr;
  }
}

void release(rbf_engine* e) {
  if (!e) return;
  if (e->stream) cudaStreamSynchronize(e->stream);
  drop_graphs(e);
  if (e->owner) {
    std::lock_guard<std::mutex> lock(e->owner->views_mu);  // the corpus belongs to the owner
    auto& v = e->owner->views;
    v.erase(std::remove(v.begin(), v.end(), e), v.end());
  } else {
    cudaFree(e->corpus);
    cudaFree(e->corpus_bf16);
  }
  cudaFree(e->query_bf16);
  cudaFree(e->query_f32);
  cudaFree(e->theta0);
  cudaFree(e->lens);
  cudaFree(e->partials);
  cudaFree(e->errw);
  cudaFree(e->counters);
  cudaFree(e->i32_theta0);
  cudaFree(e->result);
  cudaFreeHost(e->h_query);
  cudaFreeHost(e->h_result);
  if (e->own_stream && e->stream) cudaStreamDestroy(e->stream);
  delete e;
}

// RBF_FAULT=alloc: make the engine's allocations fail (tests of the
// out-of-memory path; nothing is issued to the GPU for it).
bool alloc_fault_armed() {
  const char* v = std::getenv("RBF_FAULT");
  return v && std::strcmp(v, "alloc") == 0;
}

// Every per-call buffer of an engine or a view (not the corpus). On failure
// the engine is released.
rbf_status alloc_call_buffers(rbf_engine* e) {
  bool ok = !alloc_fault_armed();
  if (e->flags & RBF_FLAG_BF16_CORPUS)
    ok = ok && cudaMalloc(&e->query_bf16, static_cast<size_t>(e->query_rows) * e->max_pitch_bf16 * 2) == cudaSuccess;
  else
    ok = ok && cudaMalloc(&e->query_f32, static_cast<size_t>(e->query_rows) * e->max_pitch * 4) == cudaSuccess;
  ok = ok && cudaMalloc(&e->theta0, static_cast<size_t>(e->max_batch) * sizeof(uint64_t)) == cudaSuccess;
  ok = ok && cudaMalloc(&e->lens, static_cast<size_t>(kBatchQueriesPerLaunch) * e->num_sms * sizeof(int)) ==
                 cudaSuccess;
  ok = ok && cudaMalloc(&e->partials, e->partials_cap * sizeof(uint64_t)) == cudaSuccess;
  ok = ok && cudaMalloc(&e->errw, 4 * sizeof(int)) == cudaSuccess;
  ok = ok && cudaMalloc(&e->counters, 8 * sizeof(unsigned)) == cudaSuccess;
  ok = ok && cudaMalloc(&e->i32_theta0, sizeof(uint64_t)) == cudaSuccess;
  ok = ok && cudaMalloc(&e->result, e->result_bytes) == cudaSuccess;
  ok = ok &&
       cudaMallocHost(&e->h_query, static_cast<size_t>(e->max_batch) * e->max_pitch * sizeof(float)) == cudaSuccess;
  ok = ok && cudaMallocHost(&e->h_result, e->result_bytes) == cudaSuccess;
  ok = ok && cudaHostGetDevicePointer(reinterpret_cast<void**>(&e->d_hres), e->h_result, 0) == cudaSuccess;
  ok = ok && cudaHostGetDevicePointer(const_cast<void**>(reinterpret_cast<const void**>(&e->d_hquery)), e->h_query,
                                      0) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    release(e);
    return RBF_ERR_OUT_OF_MEMORY;
  }
  ok = cudaMemsetAsync(e->errw, 0, 4 * sizeof(int), e->stream) == cudaSuccess &&
       cudaMemsetAsync(e->counters, 0, 8 * sizeof(unsigned), e->stream) == cudaSuccess &&
       cudaStreamSynchronize(e->stream) == cudaSuccess;
  if (!ok) {
    release(e);
    return RBF_ERR_CUDA;
  }
  return RBF_OK;
}

// A view takes its owner's corpus state (pointers, shape, readiness, corpus
// tensor map) whenever the owner has uploaded since the view last looked, and
// points its own query tensor map at its own query buffer. Its captured
// graphs are dropped then (they carry the old shape).
rbf_status sync_view(rbf_engine* e) {
  const rbf_engine* o = e->owner;
  if (!o || e->seen_version == o->corpus_version) return RBF_OK;
  cudaStreamSynchronize(e->stream);
  drop_graphs(e);
  e->corpus = o->corpus;
  e->corpus_bf16 = o->corpus_bf16;
  e->n = o->n;
  e->d = o->d;
  e->pitch = o->pitch;
  e->pitch_bf16 = o->pitch_bf16;
  e->row_offset = o->row_offset;
  e->last_lists = 0;
  e->last_k = 0;
  e->tmaps_ready = false;
  if (o->ready && o->tmaps_ready) {
    e->tmap_corpus = o->tmap_corpus;
    const bool ok = e->corpus_bf16 ? make_bf16_tensor_map(&e->tmap_query, e->query_bf16, e->query_rows, e->pitch_bf16)
                                   : make_f32_tensor_map(&e->tmap_query, e->query_f32, e->query_rows, e->pitch);
    if (!ok) return RBF_ERR_CUDA;
    e->tmaps_ready = true;
  }
  e->ready = o->ready;
  e->seen_version = o->corpus_version;
  return RBF_OK;
}

}  // namespace

extern "C" {

const char* rbf_status_string(rbf_status s) {
  switch (s) {
    case RBF_OK: return "RBF_OK";
    case RBF_ERR_INVALID_VALUE: return "RBF_ERR_INVALID_VALUE";
    case RBF_ERR_NOT_READY: return "RBF_ERR_NOT_READY";
    case RBF_ERR_OUT_OF_MEMORY: return "RBF_ERR_OUT_OF_MEMORY";
    case RBF_ERR_CUDA: return "RBF_ERR_CUDA";
    case RBF_ERR_TIMEOUT: return "RBF_ERR_TIMEOUT";
    case RBF_ERR_UNSUPPORTED: return "RBF_ERR_UNSUPPORTED";
    case RBF_ERR_BOUNDS: return "RBF_ERR_BOUNDS";
  }
  return "RBF_ERR_UNKNOWN";
}

rbf_status rbf_create(int64_t max_n, int32_t max_d, int32_t max_k, int32_t max_batch, uint32_t flags,
                      void* cuda_stream, rbf_engine** out) {
  if (!out) return RBF_ERR_INVALID_VALUE;
  if (max_n < 1 || max_n > INT32_MAX || max_d < 1 || max_d > RBF_MAX_D || max_k < 1 || max_k > RBF_MAX_K ||
      max_batch < 1 || max_batch > kMaxBatch)
    return RBF_ERR_INVALID_VALUE;
  if (flags & ~(RBF_FLAG_FP32_CORPUS | RBF_FLAG_BF16_CORPUS | RBF_FLAG_COSINE)) return RBF_ERR_INVALID_VALUE;
  if (!(flags & (RBF_FLAG_FP32_CORPUS | RBF_FLAG_BF16_CORPUS))) flags |= RBF_FLAG_FP32_CORPUS;

  rbf_engine* e = new (std::nothrow) rbf_engine();
  if (!e) return RBF_ERR_OUT_OF_MEMORY;
  cudaError_t st = cudaGetDevice(&e->device);
  if (st != cudaSuccess) {
    delete e;
    return RBF_ERR_CUDA;
  }
  cudaDeviceGetAttribute(&e->num_sms, cudaDevAttrMultiProcessorCount, e->device);
  cudaDeviceGetAttribute(&e->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, e->device);
  {
    // Address translation through the host's page tables (GB300's Grace
    // host over NVLink-C2C): a kernel may read any host buffer in place.
    int pageable = 0, host_tables = 0;
    cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, e->device);
    cudaDeviceGetAttribute(&host_tables, cudaDevAttrPageableMemoryAccessUsesHostPageTables, e->device);
    e->host_read_ok = pageable && host_tables ? 1 : 0;
    e->host_read = e->host_read_ok;
  }
  e->max_n = max_n;
  e->max_d = max_d;
  e->max_k = max_k;
  e->max_batch = max_batch;
  e->flags = flags;
  e->max_pitch = static_cast<int>(align_up(static_cast<size_t>(max_d), 4));

  if (cuda_stream) {
    e->stream = static_cast<cudaStream_t>(cuda_stream);
  } else {
    st = cudaStreamCreateWithFlags(&e->stream, cudaStreamNonBlocking);
    if (st != cudaSuccess) {
      delete e;
      return RBF_ERR_CUDA;
    }
    e->own_stream = true;
  }

  const size_t kpmax = static_cast<size_t>(list_width(max_k));
  const size_t max_lists = static_cast<size_t>(e->num_sms) * kMaxCtasPerSm;
  e->partials_cap = max_lists * kpmax;
  // Batched search: on the bf16 copy when there is one, else (tf32) on the
  // fp32 corpus itself.
  e->query_rows = static_cast<int>(align_up(static_cast<size_t>(max_batch), kBatchQueriesPerLaunch));
  const size_t batch_keys = static_cast<size_t>(max_batch) * e->num_sms * kBatchListWidth;
  e->partials_cap = std::max(e->partials_cap, batch_keys);
  // K > 32: one group of 256 queries at a time, lists of list_width(K) keys.
  if (max_k > kBatchRegMaxK)
    e->partials_cap = std::max(e->partials_cap, static_cast<size_t>(kBatchQueriesPerLaunch) * e->num_sms * kpmax);
  if (flags & RBF_FLAG_BF16_CORPUS) {
    flags |= RBF_FLAG_FP32_CORPUS;  // uploads are converted from the fp32 copy
    e->flags = flags;
    e->max_pitch_bf16 = static_cast<int>(align_up(static_cast<size_t>(max_d), kBf16PitchAlign));
  }
  const size_t result_count = static_cast<size_t>(max_batch) * max_k;
  e->result_bytes = result_layout(result_count, 8).bytes;

  bool ok = !alloc_fault_armed();
  if (flags & RBF_FLAG_FP32_CORPUS)
    ok = ok && cudaMalloc(&e->corpus, static_cast<size_t>(max_n) * e->max_pitch * sizeof(float)) == cudaSuccess;
  if (flags & RBF_FLAG_BF16_CORPUS)
    ok = ok && cudaMalloc(&e->corpus_bf16, align_up(static_cast<size_t>(max_n), 128) * e->max_pitch_bf16 * 2) ==
                   cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    release(e);
    return RBF_ERR_OUT_OF_MEMORY;
  }
  if (rbf_status st2 = alloc_call_buffers(e)) return st2;  // releases e on failure
  *out = e;
  return RBF_OK;
}

rbf_status rbf_create_view(rbf_engine* base, void* cuda_stream, rbf_engine** out) {
  if (!base || base->owner || !out) return RBF_ERR_INVALID_VALUE;
  rbf_engine* e = new (std::nothrow) rbf_engine();
  if (!e) return RBF_ERR_OUT_OF_MEMORY;
  e->device = base->device;
  e->num_sms = base->num_sms;
  e->smem_optin = base->smem_optin;
  e->max_n = base->max_n;
  e->max_d = base->max_d;
  e->max_k = base->max_k;
  e->max_batch = base->max_batch;
  e->flags = base->flags;
  e->max_pitch = base->max_pitch;
  e->max_pitch_bf16 = base->max_pitch_bf16;
  e->query_rows = base->query_rows;
  e->partials_cap = base->partials_cap;
  e->result_bytes = base->result_bytes;
  e->ctas_per_sm = base->ctas_per_sm;
  e->stage_bytes = base->stage_bytes;
  e->smem_budget = base->smem_budget;
  e->timeout_ns = base->timeout_ns;
  e->dynamic = base->dynamic;
  e->batch_sample = base->batch_sample;
  e->host_read = base->host_read;
  e->host_read_ok = base->host_read_ok;
  e->owner = base;
  e->seen_version = base->corpus_version - 1;  // read the corpus state at the first call
  try {
    std::lock_guard<std::mutex> lock(base->views_mu);
    base->views.push_back(e);
  } catch (...) {
    e->owner = nullptr;
    release(e);
    return RBF_ERR_OUT_OF_MEMORY;
  }
  if (cuda_stream) {
    e->stream = static_cast<cudaStream_t>(cuda_stream);
  } else if (cudaStreamCreateWithFlags(&e->stream, cudaStreamNonBlocking) != cudaSuccess) {
    e->stream = nullptr;
    release(e);
    return RBF_ERR_CUDA;
  } else {
    e->own_stream = true;
  }
  if (rbf_status st = alloc_call_buffers(e)) return st;
  *out = e;
  return RBF_OK;
}

rbf_status rbf_destroy(rbf_engine* e) {
  if (e) {
    std::lock_guard<std::mutex> lock(e->views_mu);
    if (!e->views.empty()) return RBF_ERR_INVALID_VALUE;
  }
  release(e);
  return RBF_OK;
}

void* rbf_stream(const rbf_engine* e) { return e ? static_cast<void*>(e->stream) : nullptr; }

int32_t rbf_num_sms(const rbf_engine* e) { return e ? e->num_sms : 0; }

int32_t rbf_num_partials(const rbf_engine* e) {
  if (!e || sync_view(const_cast<rbf_engine*>(e)) != RBF_OK || !e->ready) return 0;
  ScoreShape sh;
  return score_shape(e, 1, &sh) ? sh.grid : 0;
}

int32_t rbf_last_cuda_error(const rbf_engine* e) { return e ? e->last_cuda_error : 0; }

int32_t rbf_last_launches(const rbf_engine* e) { return e ? e->launches : 0; }

rbf_status rbf_set_option(rbf_engine* e, rbf_option opt, int64_t value) {
  if (!e) return RBF_ERR_INVALID_VALUE;
  cudaStreamSynchronize(e->stream);
  drop_graphs(e);  // captured launches carry the old launch shape
  switch (opt) {
    case RBF_OPT_CTAS_PER_SM:
      if (value < 1 || value > kMaxCtasPerSm) return RBF_ERR_INVALID_VALUE;
      e->ctas_per_sm = static_cast<int>(value);
      return RBF_OK;
    case RBF_OPT_STAGE_BYTES:
      if (value < 16 || value > (1 << 20)) return RBF_ERR_INVALID_VALUE;
      e->stage_bytes = static_cast<int>(value);
      return RBF_OK;
    case RBF_OPT_SMEM_BUDGET:
      if (value < 0 || value > e->smem_optin) return RBF_ERR_INVALID_VALUE;
      e->smem_budget = static_cast<int>(value);
      return RBF_OK;
    case RBF_OPT_TIMEOUT_NS:
      if (value < 1000) return RBF_ERR_INVALID_VALUE;
      e->timeout_ns = static_cast<uint64_t>(value);
      return RBF_OK;
    case RBF_OPT_SCHEDULE:
      if (value != 0 && value != 1) return RBF_ERR_INVALID_VALUE;
      e->dynamic = static_cast<int>(value);
      return RBF_OK;
    case RBF_OPT_BATCH_SAMPLE:
      if (value < -1 || (value > 0 && value % 256 != 0)) return RBF_ERR_INVALID_VALUE;
      e->batch_sample = value;
      return RBF_OK;
    case RBF_OPT_HOST_READ:
      if (value < 0 || value > 1) return RBF_ERR_INVALID_VALUE;
      if (value == 1 && !e->host_read_ok) return RBF_ERR_UNSUPPORTED;
      e->host_read = static_cast<int>(value);
      return RBF_OK;
  }
  return RBF_ERR_INVALID_VALUE;
}

rbf_status rbf_check_device_error(rbf_engine* e) {
  if (!e) return RBF_ERR_INVALID_VALUE;
  int w = 0;
  cudaError_t st = cudaStreamSynchronize(e->stream);
  if (st == cudaSuccess) st = cudaMemcpyAsync(&w, e->errw + 1, sizeof(int), cudaMemcpyDeviceToHost, e->stream);
  if (st == cudaSuccess) st = cudaMemsetAsync(e->errw + 1, 0, sizeof(int), e->stream);
  if (st == cudaSuccess) st = cudaStreamSynchronize(e->stream);
  if (st != cudaSuccess) return cuda_fail(e, st);
  if (w & kErrBounds) return RBF_ERR_BOUNDS;
  return w ? RBF_ERR_TIMEOUT : RBF_OK;
}

rbf_status upload_corpus_rowmajor(rbf_engine* e, const float* corpus, int64_t n, int32_t d) {
  return upload_corpus_shard(e, corpus, n, d, 0);
}

rbf_status upload_corpus_shard(rbf_engine* e, const float* corpus, int64_t n, int32_t d, int64_t row_offset) {
  if (!e || !corpus || n < 1 || n > e->max_n || d < 1 || d > e->max_d || e->owner) return RBF_ERR_INVALID_VALUE;
  if (row_offset < 0 || row_offset > int64_t(INT32_MAX) - n) return RBF_ERR_INVALID_VALUE;
  if (!e->corpus) return RBF_ERR_UNSUPPORTED;
  e->ready = false;
  ++e->corpus_version;  // views re-read the corpus state at their next call
  cudaStreamSynchronize(e->stream);
  {
    std::lock_guard<std::mutex> lock(e->views_mu);
    for (rbf_engine* v : e->views) cudaStreamSynchronize(v->stream);  // their searches in flight read the corpus
  }
  drop_graphs(e);  // captured launches carry the old corpus shape
  const int pitch = static_cast<int>(align_up(static_cast<size_t>(d), 4));
  RBF_COPY(e, cudaMemcpy2DAsync(e->corpus, static_cast<size_t>(pitch) * 4, corpus, static_cast<size_t>(d) * 4,
                                static_cast<size_t>(d) * 4, static_cast<size_t>(n), cudaMemcpyDefault, e->stream));
  if (pitch > d) {
    RBF_COPY(e, cudaMemset2DAsync(e->corpus + d, static_cast<size_t>(pitch) * 4, 0,
                                  static_cast<size_t>(pitch - d) * 4, static_cast<size_t>(n), e->stream));
  }
  if (e->flags & RBF_FLAG_COSINE)
    RBF_LAUNCH(e, launch_normalize_rows(e->corpus, n, d, pitch, e->num_sms, e->stream));
  if (e->corpus_bf16) {
    const int pb = static_cast<int>(align_up(static_cast<size_t>(d), kBf16PitchAlign));
    RBF_LAUNCH(e, launch_to_bf16_tiled(e->corpus, pitch, e->corpus_bf16, n, pb, d, e->num_sms, e->stream));
    if (!make_bf16_tiled_tensor_map(&e->tmap_corpus, e->corpus_bf16, n, pb) ||
        !make_bf16_tensor_map(&e->tmap_query, e->query_bf16, e->query_rows, pb)) {
      e->tmaps_ready = false;
      return RBF_ERR_CUDA;
    }
    e->pitch_bf16 = pb;
    e->tmaps_ready = true;
  } else {
    // tf32 batched path: tensor maps over the resident fp32 corpus and the
    // padded fp32 query buffer.
    if (!make_f32_tensor_map(&e->tmap_corpus, e->corpus, n, pitch) ||
        !make_f32_tensor_map(&e->tmap_query, e->query_f32, e->query_rows, pitch)) {
      e->tmaps_ready = false;
      return RBF_ERR_CUDA;
    }
    e->tmaps_ready = true;
  }
  cudaError_t st = cudaStreamSynchronize(e->stream);
  if (st != cudaSuccess) return cuda_fail(e, st);
  e->n = n;
  e->d = d;
  e->pitch = pitch;
  e->row_offset = row_offset;
  e->ready = true;
  e->last_lists = 0;
  e->last_k = 0;
  ++e->corpus_version;
  return RBF_OK;
}

rbf_status score_select_partials_dev(rbf_engine* e, const float* d_query, int32_t k) {
  if (!e || !d_query) return RBF_ERR_INVALID_VALUE;
  if (rbf_status s = sync_view(e)) return s;
  if (!e->ready) return RBF_ERR_NOT_READY;
  if (rbf_status s = check_k(e, k)) return s;
  e->launches = 0;
  return enqueue_score(e, d_query, k);
}

rbf_status merge_partial_topk_dev(rbf_engine* e, int32_t k, int32_t* d_idx, float* d_score) {
  if (!e || !d_idx || !d_score) return RBF_ERR_INVALID_VALUE;
  if (rbf_status s = sync_view(e)) return s;
  if (!e->ready || e->last_lists == 0) return RBF_ERR_NOT_READY;
  if (k != e->last_k) return RBF_ERR_INVALID_VALUE;
  e->launches = 0;
  return enqueue_merge(e, k, e->last_lists, 1, 0, d_idx, d_score, reinterpret_cast<int*>(e->result));
}

rbf_status search_resident_dev(rbf_engine* e, const float* d_query, int32_t k, int32_t* d_idx, float* d_score) {
  if (!e || !d_query || !d_idx || !d_score) return RBF_ERR_INVALID_VALUE;
  if (rbf_status s = sync_view(e)) return s;
  if (!e->ready) return RBF_ERR_NOT_READY;
  if (rbf_status s = check_k(e, k)) return s;
  e->launches = 0;
  bool merged = false;
  if (rbf_status s = enqueue_score(e, d_query, k, d_idx, d_score, reinterpret_cast<int*>(e->result), &merged))
    return s;
  if (merged) return RBF_OK;
  return enqueue_merge(e, k, e->last_lists, 1, 0, d_idx, d_score, reinterpret_cast<int*>(e->result));
}

// The device work of one search_resident call: scoring, with the query read
// in place from the pinned staging block (mapped; coherent over NVLink-C2C on
// GB300, ~2 us less per call than a copy node), and the merge into the pinned
// result block.
static rbf_status enqueue_host_search(rbf_engine* e, int k, const ResultLayout& L) {
  int32_t* out_idx = reinterpret_cast<int32_t*>(e->d_hres + L.a_off);
  float* out_score = reinterpret_cast<float*>(e->d_hres + L.b_off);
  int* result_err = reinterpret_cast<int*>(e->d_hres);
  bool merged = false;
  if (rbf_status s = enqueue_score(e, e->d_hquery, k, out_idx, out_score, result_err, &merged, true)) return s;
  if (merged) return RBF_OK;
  return enqueue_merge(e, k, e->last_lists, 1, 0, out_idx, out_score, result_err, true);
}

// Record enqueue_host_search for this K as a CUDA graph (one launch per
// call afterwards). Nothing is cached if anything fails.
static rbf_status capture_host_search(rbf_engine* e, int k, const ResultLayout& L) {
  cudaError_t st = cudaStreamBeginCapture(e->stream, cudaStreamCaptureModeRelaxed);
  if (st != cudaSuccess) return cuda_fail(e, st);
  const rbf_status s = enqueue_host_search(e, k, L);
  cudaGraph_t graph = nullptr;
  st = cudaStreamEndCapture(e->stream, &graph);
  if (s != RBF_OK || st != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();
    return s != RBF_OK ? s : cuda_fail(e, st);
  }
  cudaGraphExec_t exec = nullptr;
  st = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (st != cudaSuccess) return cuda_fail(e, st);
  e->host_graph[k] = exec;
  e->host_graph_lists[k] = e->last_lists;
  e->host_graph_launches[k] = e->launches;
  return RBF_OK;
}

rbf_status search_resident(rbf_engine* e, const float* query, int32_t k, int32_t* out_idx, float* out_score) {
  if (!e || !query || !out_idx || !out_score) return RBF_ERR_INVALID_VALUE;
  if (rbf_status s = sync_view(e)) return s;
  if (!e->ready) return RBF_ERR_NOT_READY;
  if (rbf_status s = check_k(e, k)) return s;
  // The query reaches the device through the pinned staging block, read in
  // place by the kernel: that is the call's copy (for fault injection).
  if (inject(e, 1)) return RBF_ERR_CUDA;
  std::memcpy(e->h_query, query, static_cast<size_t>(e->d) * 4);
  const ResultLayout L = result_layout(static_cast<size_t>(k), 4);
  e->launches = 0;
  mark_result_pending(e);
  if (!e->host_graph[k]) {
    if (rbf_status s = capture_host_search(e, k, L)) return s;
  } else {
    // One replay stands for the call's launch.
    if (inject(e, 2)) return RBF_ERR_CUDA;
    e->last_lists = e->host_graph_lists[k];
    e->last_k = k;
    e->launches = e->host_graph_launches[k];
  }
  const cudaError_t st = cudaGraphLaunch(e->host_graph[k], e->stream);
  if (st != cudaSuccess) return cuda_fail(e, st);
  if (rbf_status s = finish_host_call_polled(e)) return s;
  std::memcpy(out_idx, e->h_result + L.a_off, 4 * static_cast<size_t>(k));
  std::memcpy(out_score, e->h_result + L.b_off, 4 * static_cast<size_t>(k));
  return RBF_OK;
}

// Batched search: convert the queries to bf16, run the tensor-core scoring +
// epilogue select once per group of up to 256 queries, merge every query.
static rbf_status enqueue_batch(rbf_engine* e, const float* d_queries, int b, int k, int32_t* d_idx, float* d_score,
                                int* result_err) {
  if (!e->tmaps_ready) return RBF_ERR_NOT_READY;
  const int64_t rows_total = static_cast<int64_t>(align_up(static_cast<size_t>(b), 128));
  const bool tf32 = e->corpus_bf16 == nullptr;
  if (tf32) {
    RBF_LAUNCH(e, launch_stage_queries_f32(d_queries, e->d, e->query_f32, e->pitch, b, rows_total, e->d,
                                           (e->flags & RBF_FLAG_COSINE) != 0, e->num_sms, e->stream));
  } else if (e->flags & RBF_FLAG_COSINE) {
    RBF_LAUNCH(e, launch_normalize_queries_bf16(d_queries, e->d, e->query_bf16, e->pitch_bf16, b, rows_total, e->d,
                                                e->num_sms, e->stream));
  } else {
    RBF_LAUNCH(e, launch_to_bf16(d_queries, e->d, e->query_bf16, e->pitch_bf16, b, rows_total, e->d, e->num_sms,
                                 e->stream));
  }
  // Clusters of two CTAs over 256-row tiles: an even grid, one list per
  // query from each CTA of a pair (the CTA holds the query's TMEM lane) and
  // column half, so grid lists per query.
  auto grid_for = [&](int64_t rows) {
    const int64_t pair_tiles = (rows + 255) / 256;
    return 2 * static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(pair_tiles, e->num_sms / 2)));
  };
  // One launch of the scoring + select kernel over rows [0, rows) for the
  // queries [q0, q0 + qc) (lists at q_out0 in the partials layout).
  auto launch_group = [&](int64_t rows, int grid, int q0, int qc, int q_out0, int bound_mode, const uint64_t* theta0,
                          bool wait_inputs) -> rbf_status {
    GemmSelectLaunch a;
    a.tmap_q = &e->tmap_query;
    a.tmap_c = &e->tmap_corpus;
    a.partials = e->partials;
    a.err = e->errw;
    a.n = rows;
    a.kchunks = tf32 ? (e->d + 31) / 32 : e->pitch_bf16 / 64;
    a.tf32 = tf32 ? 1 : 0;
    a.q_row0 = q0;
    a.q_count = qc;
    a.q_out0 = q_out0;
    a.k = k;
    a.grid = grid;
    a.timeout_ns = e->timeout_ns;
    a.theta0 = theta0;
    a.bound_mode = bound_mode;
    a.lens = k > kBatchRegMaxK ? e->lens : nullptr;
    a.partials_cap = device_cap(e);
    a.lens_cap = static_cast<size_t>(kBatchQueriesPerLaunch) * e->num_sms;
    a.theta_cap = static_cast<size_t>(e->max_batch);
    // Only the first launch after the query staging waits for it before
    // streaming (after the bound merge, or another group, the queries are
    // long complete).
    a.wait_inputs = wait_inputs ? 1 : 0;
    a.index_offset = static_cast<uint32_t>(e->row_offset);
    RBF_LAUNCH(e, launch_gemm_select(a, e->stream));
    return RBF_OK;
  };
  // All groups of up to 256 queries over rows [0, rows); returns the number
  // of lists per query: in bound mode one per CTA and column half (4 keys
  // each), else one per CTA pair (32 keys each: the pair's two column halves
  // are merged in the kernel).
  auto score_groups = [&](int64_t rows, int bound_mode, const uint64_t* theta0, int* lists) -> rbf_status {
    const int grid = grid_for(rows);
    if (static_cast<size_t>(b) * grid * kBatchListWidth > e->partials_cap) return RBF_ERR_UNSUPPORTED;
    for (int q0 = 0; q0 < b; q0 += kBatchQueriesPerLaunch) {
      const int qc = std::min(kBatchQueriesPerLaunch, b - q0);
      if (rbf_status st = launch_group(rows, grid, q0, qc, q0, bound_mode, theta0,
                                       q0 == 0 && (bound_mode || theta0 == nullptr)))
        return st;
    }
    *lists = bound_mode ? grid : grid / 2;
    return RBF_OK;
  };
  // Pre-pass over the first S rows: no selection, each per-CTA list of a
  // query holds the best key of each of 4 chunks of the rows it covers, and
  // a small kernel takes the K-th largest of those chunk maxima (4 per list,
  // 512 at S = 16,384). K distinct rows score at least that much, so it is a lower
  // bound on the final K-th key, and the main pass drops every key below it.
  // About K * N / S keys pass it; above K = 32 each one costs a merge into a
  // list in global memory, so S grows with K (16,384 per 32 of K), up to a
  // quarter of the corpus.
  // The default sample is rounded up to whole rounds of 256-row tiles over
  // every CTA pair (19,456 rows on 152 SMs): the pre-pass then holds every
  // SM, so the bound kernel's small CTAs land one per SM beside it and leave
  // room for the main pass's CTAs, instead of stacking up on SMs the
  // pre-pass left free and keeping main-pass CTAs off them.
  const uint64_t* theta0 = nullptr;
  int64_t sample_rows = e->batch_sample < 0
                            ? std::min<int64_t>(kSampleRows * ((k + 31) / 32), e->n / 4 / kSampleRows * kSampleRows)
                            : std::min<int64_t>(e->batch_sample, e->n);
  if (e->batch_sample < 0 && sample_rows > 0) {
    const int64_t round_rows = static_cast<int64_t>(256) * (e->num_sms / 2);
    sample_rows = std::min<int64_t>((sample_rows + round_rows - 1) / round_rows * round_rows, e->n / 4);
  }
  if (sample_rows >= 256) {
    int lists = 0;
    if (rbf_status st = score_groups(sample_rows, 1, nullptr, &lists)) return st;
    const int total = lists * kBoundListWidth;  // chunk maxima per query, contiguous
    if (total <= RBF_KTH_MAX_KEYS) {
      RBF_LAUNCH(e, launch_kth_of_lists(e->partials, b, total, k, e->theta0, e->stream));
    } else {
      // More lists than the bound kernel takes (a device with more than 256
      // SMs): the merge kernel gives the same K-th key.
      MergeLaunch m;
      m.partials = e->partials;
      m.lists = lists;
      m.queries = b;
      m.k = k;
      m.int_keys = 0;
      m.out_a = d_idx;  // overwritten by the final merge
      m.out_b = d_score;
      m.err_call = nullptr;
      m.err_sticky = nullptr;
      m.result_err = nullptr;
      m.partials_cap = device_cap(e);
      m.kth_out = e->theta0;
      m.stride = kBoundListWidth;  // 4 chunk maxima per list
      m.short_lists = k > kBatchRegMaxK ? 1 : 0;
      RBF_LAUNCH(e, launch_merge(m, e->stream));
    }
    theta0 = e->theta0;
  }
  if (k <= kBatchRegMaxK) {
    int grid = 0;
    if (rbf_status st = score_groups(e->n, 0, theta0, &grid)) return st;
    return enqueue_merge(e, k, grid, b, 0, d_idx, d_score, result_err);
  }
  // K > 32: each group of 256 queries is scored (CTA pairs, each thread's
  // list in the partials buffer with its length in `lens`) and merged before
  // the next group reuses the buffer. The last merge hands the call's error
  // word over.
  const int grid = grid_for(e->n);
  const int kw = list_width(k);
  if (static_cast<size_t>(kBatchQueriesPerLaunch) * grid * kw > e->partials_cap) return RBF_ERR_UNSUPPORTED;
  for (int q0 = 0; q0 < b; q0 += kBatchQueriesPerLaunch) {
    const int qc = std::min(kBatchQueriesPerLaunch, b - q0);
    const bool last = q0 + qc == b;
    if (rbf_status st = launch_group(e->n, grid, q0, qc, 0, 0, theta0, q0 == 0 && theta0 == nullptr)) return st;
    MergeLaunch m;
    m.partials = e->partials;
    m.lists = grid;
    m.queries = qc;
    m.k = k;
    m.int_keys = 0;
    m.out_a = d_idx + static_cast<size_t>(q0) * k;
    m.out_b = d_score + static_cast<size_t>(q0) * k;
    m.err_call = last ? e->errw : nullptr;
    m.err_sticky = e->errw + 1;
    m.result_err = last ? result_err : nullptr;
    m.partials_cap = device_cap(e);
    m.stride = kw;
    m.lens = e->lens;
    m.short_lists = 1;
    RBF_LAUNCH(e, launch_merge(m, e->stream));
  }
  return RBF_OK;
}

rbf_status search_resident_batch_dev(rbf_engine* e, const float* d_queries, int32_t b, int32_t k, int32_t* d_idx,
                                     float* d_score) {
  if (!e || !d_queries || !d_idx || !d_score || b < 1 || b > e->max_batch) return RBF_ERR_INVALID_VALUE;
  if (rbf_status s = sync_view(e)) return s;
  if (!e->ready) return RBF_ERR_NOT_READY;
  if (rbf_status s = check_k(e, k)) return s;
  e->launches = 0;
  return enqueue_batch(e, d_queries, b, k, d_idx, d_score, reinterpret_cast<int*>(e->result));
}

rbf_status search_resident_batch(rbf_engine* e, const float* queries, int32_t b, int32_t k, int32_t* out_idx,
                                 float* out_score) {
  if (!e || !queries || !out_idx || !out_score || b < 1 || b > e->max_batch) return RBF_ERR_INVALID_VALUE;
  if (rbf_status s = sync_view(e)) return s;
  if (!e->ready) return RBF_ERR_NOT_READY;
  if (rbf_status s = check_k(e, k)) return s;
  const size_t qbytes = static_cast<size_t>(b) * e->d * 4;
  e->launches = 0;
  // The query conversion kernel reads the queries on the host (coherent over
  // NVLink-C2C on GB300): where the device reads pageable memory through the
  // host's page tables, straight from the caller's buffer (the call is
  // synchronous, so the buffer outlives every read); else from the pinned
  // staging block they are first copied into, as the single-query search
  // does. Either way that is the call's host-to-device transfer.
  if (inject(e, 1)) return RBF_ERR_CUDA;
  const float* src = queries;
  if (!e->host_read) {
    std::memcpy(e->h_query, queries, qbytes);
    src = e->d_hquery;
  }
  const size_t count = static_cast<size_t>(b) * k;
  const ResultLayout L = result_layout(count, 4);
  if (rbf_status s = enqueue_batch(e, src, b, k, reinterpret_cast<int32_t*>(e->d_hres + L.a_off),
                                   reinterpret_cast<float*>(e->d_hres + L.b_off), reinterpret_cast<int*>(e->d_hres)))
    return s;
  if (rbf_status s = finish_host_call(e, L)) return s;
  std::memcpy(out_idx, e->h_result + L.a_off, 4 * count);
  std::memcpy(out_score, e->h_result + L.b_off, 4 * count);
  return RBF_OK;
}

rbf_status merge_shard_topk_dev(rbf_engine* e, const int32_t* d_idx, const float* d_score, int32_t g, int32_t b,
                                int32_t k, int32_t* d_out_idx, float* d_out_score) {
  if (!e || !d_idx || !d_score || !d_out_idx || !d_out_score) return RBF_ERR_INVALID_VALUE;
  if (g < 1 || g > kMaxShards || b < 1 || b > e->max_batch || k < 1 || k > e->max_k) return RBF_ERR_INVALID_VALUE;
  const int kp = list_width(k);
  if (static_cast<size_t>(b) * g * kp > e->partials_cap) return RBF_ERR_UNSUPPORTED;
  e->launches = 0;
  e->last_lists = 0;  // the partials buffer is reused: a pending two-step merge is void
  RBF_LAUNCH(e, launch_encode_shard_lists(d_idx, d_score, g, b, k, kp, e->partials, e->num_sms, e->stream));
  MergeLaunch m;
  m.partials = e->partials;
  m.lists = g;
  m.queries = b;
  m.k = k;
  m.int_keys = 0;
  m.out_a = d_out_idx;
  m.out_b = d_out_score;
  m.err_call = e->errw;
  m.err_sticky = e->errw + 1;
  m.result_err = reinterpret_cast<int*>(e->result);
  m.partials_cap = device_cap(e);
  m.stride = kp;
  RBF_LAUNCH(e, launch_merge(m, e->stream));
  return RBF_OK;
}

static rbf_status enqueue_topk_int32(rbf_engine* e, const int32_t* d_data, int64_t n, int32_t k, int32_t* val,
                                     int64_t* pos, int* result_err, bool host_result = false) {
  // Register-load stage 1 over contiguous ranges; below 8,192 elements per
  // CTA fewer CTAs are used.
  auto stage1 = [&](int64_t count, int* lists) -> rbf_status {
    const int64_t per_cta = 8192;
    int64_t grid = std::min<int64_t>(int64_t(e->num_sms) * kI32CtasPerSm, (count + per_cta - 1) / per_cta);
    grid = std::max<int64_t>(grid, 1);
    if (static_cast<size_t>(grid) * list_width(k) > e->partials_cap) return RBF_ERR_UNSUPPORTED;
    I32Launch a;
    a.data = d_data;
    a.n = count;
    a.k = k;
    a.partials = e->partials;
    a.partials_cap = device_cap(e);
    a.err = e->errw;
    a.grid = static_cast<int>(grid);
    RBF_LAUNCH(e, launch_topk_i32_stage1(a, e->stream));
    *lists = static_cast<int>(grid);
    return RBF_OK;
  };
  int lists = 0;
  if (n < kI32StreamMin) {
    if (rbf_status st = stage1(n, &lists)) return st;
    return enqueue_merge(e, k, lists, 1, 1, val, pos, result_err, host_result);
  }
  // Large arrays: the bulk-copy ring kernel, one CTA per SM. Each CTA bounds
  // the K-th key from its own slice before its first tile. That bound weakens
  // as K grows (it comes from 32,768 values), so for K >= kI32SampleMinK the
  // exact K-th key of the first kI32SampleElems elements -- also a lower
  // bound, as they are part of the array -- is computed first and passed in.
  if (static_cast<size_t>(e->num_sms) * list_width(k) > e->partials_cap) return RBF_ERR_UNSUPPORTED;
  const uint64_t* theta0 = nullptr;
  if (k >= kI32SampleMinK) {
    int sample_lists = 0;
    if (rbf_status st = stage1(kI32SampleElems, &sample_lists)) return st;
    MergeLaunch m;
    m.partials = e->partials;
    m.lists = sample_lists;
    m.queries = 1;
    m.k = k;
    m.int_keys = 1;
    m.out_a = val;  // overwritten by the final merge
    m.out_b = pos;
    m.err_call = nullptr;
    m.err_sticky = nullptr;
    m.result_err = nullptr;
    m.partials_cap = device_cap(e);
    m.kth_out = e->i32_theta0;
    RBF_LAUNCH(e, launch_merge(m, e->stream));
    theta0 = e->i32_theta0;
  }
  I32StreamLaunch a;
  a.data = d_data;
  a.n = n;
  a.k = k;
  a.partials = e->partials;
  a.partials_cap = device_cap(e);
  a.theta0 = theta0;
  a.counters = e->counters + 2;
  a.err = e->errw;
  a.grid = e->num_sms;
  a.timeout_ns = e->timeout_ns;
  // Stage 2 runs in the kernel's last CTA.
  a.out_val = val;
  a.out_pos = pos;
  a.err_sticky = e->errw + 1;
  a.result_err = result_err;
  a.host_result = host_result ? 1 : 0;
  RBF_LAUNCH(e, launch_topk_i32_stream(a, e->stream));
  return RBF_OK;
}

static rbf_status check_i32_args(const rbf_engine* e, const int32_t* d_data, int64_t n, int32_t k) {
  if (!e || !d_data || n < 1 || n > int64_t(0xFFFFFFFFll)) return RBF_ERR_INVALID_VALUE;
  if (k < 1 || k > e->max_k || static_cast<int64_t>(k) > n) return RBF_ERR_INVALID_VALUE;
  if ((reinterpret_cast<uintptr_t>(d_data) & 3u) != 0) return RBF_ERR_INVALID_VALUE;
  return RBF_OK;
}

rbf_status topk_int32_dev(rbf_engine* e, const int32_t* d_data, int64_t n, int32_t k, int32_t* d_val,
                          int64_t* d_pos) {
  if (rbf_status s = check_i32_args(e, d_data, n, k)) return s;
  if (!d_val || !d_pos) return RBF_ERR_INVALID_VALUE;
  e->launches = 0;
  return enqueue_topk_int32(e, d_data, n, k, d_val, d_pos, reinterpret_cast<int*>(e->result));
}

rbf_status topk_int32(rbf_engine* e, const int32_t* d_data, int64_t n, int32_t k, int32_t* out_val,
                      int64_t* out_pos) {
  if (rbf_status s = check_i32_args(e, d_data, n, k)) return s;
  if (!out_val || !out_pos) return RBF_ERR_INVALID_VALUE;
  const ResultLayout L = result_layout(static_cast<size_t>(k), 8);
  e->launches = 0;
  mark_result_pending(e);
  if (rbf_status s = enqueue_topk_int32(e, d_data, n, k, reinterpret_cast<int32_t*>(e->d_hres + L.a_off),
                                        reinterpret_cast<int64_t*>(e->d_hres + L.b_off),
                                        reinterpret_cast<int*>(e->d_hres), true))
    return s;
  if (rbf_status s = finish_host_call_polled(e)) return s;
  std::memcpy(out_val, e->h_result + L.a_off, 4 * static_cast<size_t>(k));
  std::memcpy(out_pos, e->h_result + L.b_off, 8 * static_cast<size_t>(k));
  return RBF_OK;
}

rbf_status rbf_selftest_wait_timeout(rbf_engine* e, uint64_t timeout_ns) {
  if (!e || timeout_ns < 1000 || timeout_ns > 10000000000ull) return RBF_ERR_INVALID_VALUE;
  RBF_COPY(e, cudaMemsetAsync(e->errw + 2, 0, sizeof(int), e->stream));
  RBF_LAUNCH(e, launch_wait_probe(e->errw + 2, timeout_ns, e->stream));
  int w = 0;
  RBF_COPY(e, cudaMemcpyAsync(&w, e->errw + 2, sizeof(int), cudaMemcpyDeviceToHost, e->stream));
  cudaError_t st = cudaStreamSynchronize(e->stream);
  if (st != cudaSuccess) return cuda_fail(e, st);
  return w ? RBF_ERR_TIMEOUT : RBF_OK;
}

rbf_status rbf_inject_host_fault(rbf_engine* e, int32_t kind, int32_t count) {
  if (!e || count < 0 || (count > 0 && kind != 1 && kind != 2)) return RBF_ERR_INVALID_VALUE;
  e->fault_kind = kind;
  e->fault_count = count;
  return RBF_OK;
}

}  // extern "C"
