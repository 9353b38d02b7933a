/*
 * rbf.h -- C ABI of the GB300 resident brute-force top-K library (librbf.so).
 *
 * Exact top-K retrieval over a corpus that stays in GPU memory: a query of D
 * floats is scored by inner product against N corpus rows, and the K rows
 * with the highest scores come back best-first (GPU-Resident Top-K for
 * Agentic RAG, section 2 and the "architecture mental model" pipeline:
 * query up, score, per-block partial top-K, merge, K indices + K scores down).
 *
 * Ordering rule used by every entry point (same article, section 3, problem
 * B): a higher score is better; on an exactly equal fp32 score the lower row
 * index is better. -0.0 and +0.0 are equal; a NaN score ranks as -infinity.
 * Results are always best-first.
 *
 * Conventions
 *   - All sizes are element counts. Matrices are dense row-major.
 *   - "host" pointers are ordinary CPU memory (pageable or pinned);
 *     "device" pointers are CUDA device memory on the engine's device.
 *   - The caller owns every pointer it passes; the library keeps none of them
 *     after the call returns.
 *   - The engine owns all device memory it uses. It is allocated in
 *     rbf_create and nothing is allocated afterwards (the article's "engine
 *     initialise" step, section 3 problem C and section 4 step 0).
 *   - Calls ending in _dev are stream-ordered on the engine's stream: they
 *     enqueue work and return; their outputs are valid once that stream has
 *     reached them. The other calls are synchronous.
 *   - Errors are returned, never thrown. On any error the caller's output
 *     buffers are left untouched. RBF_ERR_CUDA records the CUDA error code,
 *     readable with rbf_last_cuda_error.
 *   - One engine is not safe for concurrent calls from several host threads;
 *     callers serialise (the article's own caveat, section 9).
 */
#ifndef RBF_H_
#define RBF_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct rbf_engine rbf_engine;

typedef enum rbf_status {
  RBF_OK = 0,
  RBF_ERR_INVALID_VALUE = 1, /* bad size, K, pointer or flag */
  RBF_ERR_NOT_READY = 2,     /* search before any corpus upload */
  RBF_ERR_OUT_OF_MEMORY = 3, /* rbf_create could not allocate */
  RBF_ERR_CUDA = 4,          /* a CUDA runtime call failed */
  RBF_ERR_TIMEOUT = 5,       /* a bounded device-side wait ran out */
  RBF_ERR_UNSUPPORTED = 6,   /* valid request beyond the engine's launch limits */
  RBF_ERR_BOUNDS = 7         /* checked builds (RBF_CHECKS) only: a kernel met an index outside
                                its buffer and skipped the access; the outputs are not valid */
} rbf_status;

/* Largest K any entry point accepts (the article's kMaxSupportedK,
 * section 4 step 3). */
#define RBF_MAX_K 256
/* Largest embedding width D. */
#define RBF_MAX_D 8192

/* rbf_create flags. 0 means RBF_FLAG_FP32_CORPUS. */
#define RBF_FLAG_FP32_CORPUS 0x1u /* keep the fp32 corpus: single-query path */
#define RBF_FLAG_BF16_CORPUS 0x2u /* also keep a bf16 copy for the batched path (else it runs tf32) */
/* Score by cosine similarity instead of the inner product: the inner product
 * divided by the product of the query's and the row's L2 norms, and -infinity
 * for a row whose denominator is not positive (GPU-Resident Top-K for Agentic
 * RAG, section 4 step 2, the scoring kernel's cosine mode). Rows are divided
 * by their norms once at upload (the stored corpus is the normalised one) and
 * every query at every call, as the same article suggests; a zero-norm row or
 * query scores -infinity everywhere. Applies to every float search entry
 * point of the engine; topk_int32 is unaffected. */
#define RBF_FLAG_COSINE 0x4u

/* Engine options for rbf_set_option (launch shape of the scoring kernel). */
typedef enum rbf_option {
  RBF_OPT_CTAS_PER_SM = 1,   /* persistent CTAs per SM, 1..4 (default 1) */
  RBF_OPT_STAGE_BYTES = 2,   /* target bytes per pipeline stage (default 65536) */
  RBF_OPT_SMEM_BUDGET = 3,   /* shared-memory ring budget per CTA, bytes */
  RBF_OPT_TIMEOUT_NS = 4,    /* bound on every device-side wait (default 2e9) */
  RBF_OPT_SCHEDULE = 5,      /* 0 = static row ranges, 1 = dynamic tile claims (default) */
  RBF_OPT_BATCH_SAMPLE = 6,  /* rows of the batched path's bound pre-pass: -1 = automatic
                                (default: 16,384 per 32 of K, at most N/4 and none below
                                N = 65,536, rounded up to whole rounds of 256-row tiles over
                                every CTA pair), 0 = no pre-pass, else that many leading rows (a
                                multiple of 256, at most N). Changes speed only, never results. */
  RBF_OPT_HOST_READ = 7      /* 1 = search_resident_batch's first kernel reads the caller's
                                query buffer in place (the default where the device reads pageable
                                host memory through the host's page tables, as a GB300 with its
                                Grace host does over NVLink-C2C; UNSUPPORTED elsewhere); 0 = the
                                queries are first copied into the engine's pinned staging block.
                                Changes speed only, never results. */
} rbf_option;

/* ------------------------------------------------------------------ engine */

/* Create an engine on the current CUDA device and allocate everything it will
 * ever use, sized for the worst case (max_n rows, max_d columns, max_k results,
 * max_batch queries per batched call).
 *   max_n      1 .. 2^31-1
 *   max_d      1 .. RBF_MAX_D
 *   max_k      1 .. RBF_MAX_K
 *   max_batch  1 .. 4096 (>= 1 even if only single queries are used)
 *   flags      RBF_FLAG_* (0 = fp32 corpus only)
 *   cuda_stream  a cudaStream_t to run on, or NULL for an engine-owned
 *                non-blocking stream. A caller stream must outlive the engine.
 *   out        receives the engine handle.
 * Errors: INVALID_VALUE (a size out of range, out == NULL),
 *         OUT_OF_MEMORY (device or pinned-host allocation failed),
 *         CUDA (no usable device). */
rbf_status rbf_create(int64_t max_n, int32_t max_d, int32_t max_k, int32_t max_batch,
                      uint32_t flags, void* cuda_stream, rbf_engine** out);

/* A second handle on `base`'s resident corpus, with its own stream and its
 * own per-call buffers (partial lists, counters, error words, query staging,
 * pinned result block, captured graphs) but no copy of the corpus: calls on
 * different handles of one corpus may run at the same time, from different
 * host threads and on different streams. One engine alone is not safe for
 * concurrent calls (GPU-Resident Top-K for Agentic RAG, section 9, names
 * that as a limitation; CUDA programming model series 9, section 4.2, runs
 * independent top-K work on separate streams). The view takes the base's
 * sizes, flags and options; set_option on a view changes only the view.
 * An upload on the base first waits for the work already queued on its views'
 * streams, and its views see the new corpus at their next call; the upload
 * call itself must not run at the same time as a call on a view (from another
 * host thread). Views cannot upload. Views may be made and destroyed from
 * any host thread, also while other views of the same base are in use.
 *   base         an engine made by rbf_create (not a view)
 *   cuda_stream  a cudaStream_t, or NULL for a view-owned non-blocking stream
 *   out          receives the view handle (destroy it with rbf_destroy,
 *                before the base)
 * Errors: INVALID_VALUE (base NULL or a view, out NULL), OUT_OF_MEMORY, CUDA. */
rbf_status rbf_create_view(rbf_engine* base, void* cuda_stream, rbf_engine** out);

/* Synchronise the engine's stream and free everything it owns. NULL is a no-op.
 * Errors: INVALID_VALUE (an engine that still has views). */
rbf_status rbf_destroy(rbf_engine* engine);

/* The cudaStream_t the engine runs on. */
void* rbf_stream(const rbf_engine* engine);

/* Number of SMs of the engine's device. */
int32_t rbf_num_sms(const rbf_engine* engine);

/* Number of per-CTA partial lists the scoring step writes for the resident
 * corpus (0 before an upload). */
int32_t rbf_num_partials(const rbf_engine* engine);

/* Change a launch option (see rbf_option); takes effect on the next call. */
rbf_status rbf_set_option(rbf_engine* engine, rbf_option option, int64_t value);

/* Human-readable name of a status code (static string). */
const char* rbf_status_string(rbf_status status);

/* cudaError_t value of the most recent RBF_ERR_CUDA on this engine. */
int32_t rbf_last_cuda_error(const rbf_engine* engine);

/* Number of kernels the engine's most recent search or top-K call enqueued
 * (a replayed graph counts the kernels captured in it); 0 before any call. */
int32_t rbf_last_launches(const rbf_engine* engine);

/* Synchronise the stream and return (and clear) any error a device kernel
 * recorded since the last check: RBF_ERR_TIMEOUT if a bounded wait ran out,
 * RBF_ERR_BOUNDS if a checked build skipped an access outside its buffer. */
rbf_status rbf_check_device_error(rbf_engine* engine);

/* ------------------------------------------------------------------ ingest */

/* Copy a row-major N x D fp32 corpus into the engine and make it resident
 * (the article's upload_corpus_rowmajor, section 4 step 1). corpus may be a
 * host or a device pointer. Rows are stored with a pitch rounded up to a
 * multiple of 4 floats and zero-padded; with RBF_FLAG_BF16_CORPUS a bf16 copy
 * (round-to-nearest-even) is made too. A new upload replaces the old corpus.
 * Blocks until the copy is complete.
 * Errors: INVALID_VALUE (N < 1, N > max_n, D < 1, D > max_d, corpus NULL, a
 * view). */
rbf_status upload_corpus_rowmajor(rbf_engine* engine, const float* corpus, int64_t n, int32_t d);

/* Row shard of a larger corpus: as upload_corpus_rowmajor, for the rows
 * [row_offset, row_offset + n) of a row-major corpus too large for one
 * engine (GPU-Resident Top-K for Agentic RAG, section 4 step 1 and section
 * 9: past one GPU's memory the corpus is split across GPUs). Every search
 * call of the engine (and of its views) then reports global row indices,
 * local row + row_offset, and breaks exact score ties by the global index, so
 * that merge_shard_topk_dev over the shards' results gives exactly what one
 * engine holding the whole corpus would. upload_corpus_rowmajor is this call
 * with row_offset 0.
 *   row_offset  0 .. 2^31-1 - n (global indices must fit in int32)
 * Errors: those of upload_corpus_rowmajor, INVALID_VALUE (row_offset out of
 * range). */
rbf_status upload_corpus_shard(rbf_engine* engine, const float* corpus, int64_t n, int32_t d, int64_t row_offset);

/* ---------------------------------------------------------- single query */

/* Top-K of one query against the resident corpus (the article's
 * search_resident, section 4 steps 2-6: query to the device, scoring,
 * per-block partial top-K, merge, results back). Here the query is copied
 * into the engine's pinned staging block, which the scoring kernel reads in
 * place; one launch scores every row, keeps per-CTA top-K lists and merges
 * them in its last CTA, writing the K results straight into the pinned
 * result block; the call returns after synchronising the engine's stream.
 * The launch is a CUDA graph captured on the first call for each k.
 *   query      host, D floats (D of the resident corpus)
 *   k          1 .. min(max_k, N)
 *   out_idx    host, K int32 row indices, best-first
 *   out_score  host, K fp32 scores (fp32 accumulation of the inner product)
 * Errors: INVALID_VALUE, NOT_READY, CUDA, TIMEOUT. */
rbf_status search_resident(rbf_engine* engine, const float* query, int32_t k, int32_t* out_idx,
                           float* out_score);

/* As search_resident, with the query and outputs in device memory,
 * stream-ordered. d_query needs no alignment beyond 4 bytes. */
rbf_status search_resident_dev(rbf_engine* engine, const float* d_query, int32_t k, int32_t* d_idx,
                               float* d_score);

/* Step 1 of search_resident_dev alone: score every resident row against
 * d_query and leave one best-first top-K list per CTA in the engine's
 * workspace (the article's scoring and per-block partial top-K steps,
 * section 4 steps 2-3, fused so the N scores never reach memory).
 * Stream-ordered. */
rbf_status score_select_partials_dev(rbf_engine* engine, const float* d_query, int32_t k);

/* Step 2 of search_resident_dev alone: merge the per-CTA lists left by the
 * last score_select_partials_dev into the global top-K (the article's merge
 * step, section 4 step 4), same k. Stream-ordered; outputs in device memory. */
rbf_status merge_partial_topk_dev(rbf_engine* engine, int32_t k, int32_t* d_idx, float* d_score);

/* ---------------------------------------------------------------- batched */

/* Top-K of each of B queries (row-major B x D) against the resident corpus,
 * with the scoring on the tensor cores and the selection fused into their
 * epilogue (the same per-block partial top-K and merge as the single-query
 * path, GPU-Resident Top-K for Agentic RAG, section 4 steps 2-4). With
 * RBF_FLAG_BF16_CORPUS scores are bf16 x bf16 products (queries rounded to
 * bf16 on the device) accumulated in fp32; without it the resident fp32
 * corpus and fp32 queries are multiplied as tf32 (10-bit mantissas),
 * accumulated in fp32.
 *   queries    host, B x D floats
 *   b          1 .. max_batch
 *   k          1 .. min(max_k, N). Up to 32 each epilogue thread keeps its
 *              list in registers; above 32 (at most 256) in the engine's
 *              preallocated partials buffer, 256 queries at a time.
 *   out_idx    host, B x K int32 (row q holds query q's list, best-first)
 *   out_score  host, B x K fp32
 * The call is synchronous. Where the device reads pageable host memory
 * through the host's page tables (RBF_OPT_HOST_READ, on by default there) its
 * first kernel reads `queries` in place, so the buffer must be ordinary host
 * memory the process can read; otherwise the queries are copied into the
 * engine's pinned staging block first. The outputs are written only on
 * success.
 * Errors: INVALID_VALUE, NOT_READY, CUDA, TIMEOUT. */
rbf_status search_resident_batch(rbf_engine* engine, const float* queries, int32_t b, int32_t k,
                                 int32_t* out_idx, float* out_score);

/* As search_resident_batch with device queries and outputs, stream-ordered. */
rbf_status search_resident_batch_dev(rbf_engine* engine, const float* d_queries, int32_t b,
                                     int32_t k, int32_t* d_idx, float* d_score);

/* ------------------------------------------------------- row shards */

/* Merge the results of g row shards into the global top-K of each of b
 * queries: the article's merge step (section 4 step 4) applied across GPUs
 * instead of across CTAs, after the exchange of every shard's K best
 * (section 9 lists sharding across GPUs as the way past one GPU's memory).
 * Each shard's list is what search_resident(_dev) or search_resident_batch
 * (_dev) returned on an engine loaded with upload_corpus_shard (global
 * indices, best-first); entries with a negative index are missing (a shard
 * with fewer than K rows) and rank last. The shards must be disjoint row
 * ranges, so that no index appears twice. The result is best-first under the
 * ordering rule; if the shards hold fewer than K rows in all, the last
 * entries are index -1 with a NaN score.
 *   d_idx      device, [g][b][k] int32: shard s's list for query q at
 *              (s * b + q) * k (the layout an all-gather of every shard's
 *              [b][k] result produces)
 *   d_score    device, [g][b][k] fp32, the matching scores
 *   g          1 .. 1024 shards
 *   b          1 .. max_batch queries
 *   k          1 .. max_k
 *   d_out_idx  device, [b][k] int32
 *   d_out_score device, [b][k] fp32
 * Stream-ordered on the engine's stream (two launches: the lists become
 * keys in the engine's partials buffer, then the merge kernel); needs no
 * resident corpus. Errors: INVALID_VALUE, UNSUPPORTED (b * g * list width
 * beyond the partials buffer), CUDA. */
rbf_status merge_shard_topk_dev(rbf_engine* engine, const int32_t* d_idx, const float* d_score, int32_t g,
                                int32_t b, int32_t k, int32_t* d_out_idx, float* d_out_score);

/* ---------------------------------------------------------- flat int32 */

/* The K largest values of a flat int32 array in device memory, with their
 * positions, largest first, lower position first among equal values
 * (CUDA programming model series 9: stage 1 per-CTA top-K over a grid-stride
 * share of the array, section 2; stage 2 one CTA over the GRID x K
 * candidates, section 3.1).
 *   d_data   device, n int32 (4-byte aligned; no other alignment needed)
 *   n        1 .. 2^32-1
 *   k        1 .. min(max_k, n)
 *   out_val  host, K int32
 *   out_pos  host, K int64
 * Synchronous. Errors: INVALID_VALUE, CUDA, TIMEOUT. */
rbf_status topk_int32(rbf_engine* engine, const int32_t* d_data, int64_t n, int32_t k,
                      int32_t* out_val, int64_t* out_pos);

/* As topk_int32 with device outputs, stream-ordered. */
rbf_status topk_int32_dev(rbf_engine* engine, const int32_t* d_data, int64_t n, int32_t k,
                          int32_t* d_val, int64_t* d_pos);

/* No-allocation variant of topk_int32_dev, for callers that may not call
 * cudaMalloc: for example a plugin inside an inference server or database
 * whose GPU memory all comes from the host application's allocator (a
 * cudaMalloc behind its back breaks that accounting and can synchronise the
 * device, stalling the application's other streams), or latency-critical
 * code that cannot wait for an allocation. The retrieval pages have no
 * counterpart to this entry point.
 *
 * Needs no engine. It gives the same result as topk_int32_dev, computed by
 * the register-load stage-1 kernel (at most 512 CTAs, each keeping a top-K of
 * a contiguous range) followed by the merge kernel. That is the pair
 * topk_int32_dev uses below 262,144 elements; from that size on
 * topk_int32_dev runs the one-launch bulk-copy stream kernel instead, which
 * this entry point does not, so it is slower on large arrays. Neither of its
 * two kernels waits on anything, so no call can time out. Their only scratch
 * (one 256-key list per stage-1 CTA, at most 512 lists) is a fixed 1 MiB
 * array in the library's own device memory, which every GPU that loads the
 * library keeps until the process exits. The call allocates and frees
 * nothing, and calls no allocating library routine; the array's memory is
 * committed when the library's device code is loaded on a device, which with
 * CUDA's lazy module loading (the default) can happen inside the first call
 * on that device and may synchronise it, so make that first call at set-up.
 *   d_data    device, n int32 (4-byte aligned), on the current device
 *   n         1 .. 2^32-1
 *   k         1 .. min(RBF_MAX_K, n); a larger k is rejected with
 *             RBF_ERR_INVALID_VALUE (the scratch lists hold 256 keys)
 *   d_val     device, K int32, largest first
 *   d_pos     device, K int64 positions
 *   cuda_stream  stream to enqueue on (NULL = legacy default stream)
 * Stream-ordered; returns once both kernels are enqueued.
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it; make that first call before any
 * stream capture. Every call shares the one array and it keeps the previous
 * call's contents; each call writes every list it reads, so nothing needs
 * clearing, but calls whose kernels overlap on the GPU (two streams, or two
 * host threads) race on the array: serialise them. The checked build
 * (RBF_CHECKS) cannot report a skipped out-of-bounds access here, as there is
 * no error word to report it through.
 * Errors: INVALID_VALUE (arguments), CUDA (lookup or launch failed). */
rbf_status topk_int32_noalloc(const int32_t* d_data, int64_t n, int32_t k, int32_t* d_val, int64_t* d_pos,
                              void* cuda_stream);

/* ------------------------------------------------------------ self-test */

/* Launch a one-block kernel that waits, with the engine's bounded-wait
 * routine, on an mbarrier nothing ever arrives at, for at most timeout_ns.
 * Returns RBF_ERR_TIMEOUT when the wait ran out and the kernel reported it
 * (the expected outcome), RBF_OK if it somehow completed. The GPU context
 * stays usable either way. */
rbf_status rbf_selftest_wait_timeout(rbf_engine* engine, uint64_t timeout_ns);

/* Host-side fault injection for tests: the next `count` CUDA operations of the
 * given kind report failure without being issued. kind: 1 = copy, 2 = kernel
 * launch. count 0 clears. Touches no GPU state. Allocation failures are
 * injected through the environment instead (there is no engine yet): with
 * RBF_FAULT=alloc set, rbf_create and rbf_create_view fail with
 * RBF_ERR_OUT_OF_MEMORY as if a device allocation had failed, after freeing
 * what they had allocated. */
rbf_status rbf_inject_host_fault(rbf_engine* engine, int32_t kind, int32_t count);

#ifdef __cplusplus
}
#endif

#endif /* RBF_H_ */
