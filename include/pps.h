/*
 * pps.h -- C ABI of the paged, prefix-shared, mixed-batch attention library
 * (libpps.so, hand-written CUDA for sm_103a).
 *
 * The library computes, for one batch that mixes prefill chunks, single-token
 * decode rows and multi-token speculative-verify rows, exact causal GQA
 * attention over a paged KV cache whose pages may be shared between requests
 * by a radix-tree prefix cache:
 *
 *   o[r, j, h] = sum_{p <= c_r + j} softmax_p(scale * q[r, j, h] . k[r, p, h / G]) v[r, p, h / G]
 *
 * for every request r, new token j (absolute position c_r + j, c_r = tokens
 * cached before the step) and query head h, G = num_q_heads / num_kv_heads.
 * Verify rows may also form a draft tree (pps_attn_plan_tree): a draft token
 * then sees the cached positions, its ancestors and itself.
 *
 * Around that path the library also provides the steps that feed it and the
 * GEMMs of the same batch:
 *  - pps_cache_*   host radix-tree prefix cache + page allocator producing the
 *                  page tables (token-wise reuse, copy-on-write via
 *                  pps_copy_slots, LRU / LFU eviction);
 *  - pps_sched_*   token-wise budget scheduler forming each step's batch;
 *  - pps_gemm_bf16 virtual-padded projection GEMM for the batch's token rows.
 *
 * Sources (page title and section):
 *  - XY-Serve review, "Tackling the Dynamicity in a Production LLM Serving
 *    System with SOTA Optimizations via Hybrid Prefill/Decode/Verify
 *    Scheduling on Efficient Meta-kernels" (pith.science/paper/ABCKJ6RF):
 *    "Core claim" (token-budgeted P/D/V batch; workload decomposition into
 *    tile tasks recorded in token and task tables; one matmul-softmax-matmul
 *    meta-kernel; mask sparsity skips invalid tiles), "What carries the
 *    argument" (tiles sorted by computational area and assigned to cores
 *    symmetrically round-robin), "Assumptions & free parameters" (PagedAttention
 *    block table with radix-tree reuse and copy-on-write; online softmax equals
 *    plain softmax; padded scores excluded).
 *  - SGLang review, "SGLang: Efficient Execution of Structured Language Model
 *    Programs" (pith.science/p/2312.07104), "Core claim": RadixAttention reuses
 *    the KV cache of shared prefixes across requests.
 *
 * Conventions for every call:
 *  - bf16 means IEEE bfloat16 (2 bytes), little endian.  All tensors are dense
 *    and row-major with the shapes given; no strides are accepted.
 *  - "device" pointers point to memory of the current CUDA device; "host"
 *    pointers to ordinary (pageable or pinned) host memory.
 *  - The caller owns every buffer it passes.  The library keeps no pointer to
 *    them after a call returns, except that work it enqueued on `stream` still
 *    reads/writes them until that work completes.
 *  - Calls never throw and never abort.  They return PPS_OK (0) or a negative
 *    pps_status.  Argument errors are detected on the host before anything is
 *    enqueued.  Errors that only the GPU can see (a page id read from a device
 *    array that is out of range) are recorded in a device error word: the
 *    device's own (pps_get_device_error), or the one the caller registered for
 *    the stream the work runs on (pps_set_stream_error_word).  Kernels never
 *    trap.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Work is enqueued asynchronously on it.
 *  - Supported shapes: head_dim in {64, 128}; page_size in {16, 32, 64, 128};
 *    G = num_q_heads / num_kv_heads in {1, 2, 4, 8}.
 */
#ifndef PPS_H_
#define PPS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t pps_status;

#define PPS_OK 0
#define PPS_ERR_INVALID_ARGUMENT (-1)  /* null pointer, negative size, mismatched shapes   */
#define PPS_ERR_UNSUPPORTED (-2)       /* head_dim / page_size / G outside the supported set */
#define PPS_ERR_PAGE_TABLE (-3)        /* indptr not monotone, page list too short, id out of range */
#define PPS_ERR_WORKSPACE (-4)         /* workspace null or smaller than the plan requires  */
#define PPS_ERR_CUDA (-5)              /* a CUDA runtime/driver call failed                 */
#define PPS_ERR_NO_MEMORY (-6)         /* host allocation failed                            */
#define PPS_ERR_SCRATCH_LIMIT (-7)     /* plan needs more than the fixed no-alloc scratch    */
#define PPS_ERR_CACHE_FULL (-8)        /* prefix cache: no free page and nothing evictable   */

/* Device error word values (pps_get_device_error).  0 = no error. */
#define PPS_DEV_ERR_APPEND_PAGE_ID 1     /* kv_append read a page id outside [0, num_pages)   */
#define PPS_DEV_ERR_APPEND_PAGE_LIST 2   /* kv_append position beyond the request's page list */
#define PPS_DEV_ERR_APPEND_REQUEST 3     /* kv_append token not inside q_indptr's range       */
#define PPS_DEV_ERR_WAIT_TIMEOUT 4       /* a bounded pipeline wait in a kernel ran out       */
#define PPS_DEV_ERR_COPY_ARGUMENT 5      /* copy_slots: page id or slot count out of range    */

/*
 * The paged KV pool: two caller-owned device arrays, bf16,
 * [num_pages, num_kv_heads, page_size, head_dim] (all slots of one page and
 * one kv head are contiguous: page_size * head_dim * 2 bytes).
 * Logical position p of request r lives in page
 * page_indices[page_indptr[r] + p / page_size], slot p % page_size
 * (PagedAttention block table; XY-Serve review, "Assumptions & free
 * parameters").  Requests that share a cached prefix list the same page ids.
 */
typedef struct pps_pool {
  void* k;
  void* v;
  int32_t num_pages;
  int32_t num_kv_heads;
  int32_t page_size;
  int32_t head_dim;
} pps_pool;

/*
 * pps_kv_append -- write this step's new K/V rows into their pool pages.
 *
 * New token j of request r (row q_indptr[r] + j of k_new / v_new) goes to
 * logical position cached_len[r] + j.  Definition: the paged block table of
 * the XY-Serve review ("Assumptions & free parameters") with chunked-prefill,
 * decode and verify rows appended the same way ("Core claim").
 *
 *  pool          host pointer to the pool descriptor (its k/v are device).
 *  k_new, v_new  device, bf16 [num_new_tokens, num_kv_heads, head_dim].
 *  q_indptr      device int32 [num_requests + 1], q_indptr[0] = 0, nondecreasing,
 *                q_indptr[num_requests] = num_new_tokens.
 *  cached_len    device int32 [num_requests].
 *  page_indptr   device int32 [num_requests + 1]; page_indices device int32 [nnz].
 * The copy is bit exact.  Because the tables are device arrays the host only
 * checks sizes and pointers; a page id or position out of range is skipped
 * and recorded in the device error word (PPS_DEV_ERR_APPEND_*).
 * Rows of different requests must not map to the same slot (undefined order).
 */
pps_status pps_kv_append(const pps_pool* pool, const void* k_new, const void* v_new,
                         const int32_t* q_indptr, const int32_t* cached_len,
                         const int32_t* page_indptr, const int32_t* page_indices,
                         int32_t num_requests, int32_t num_new_tokens, void* stream);

/*
 * pps_copy_slots -- copy-on-write of partly reused pages: for each i < count,
 * slots [0, num_slots[i]) of page src_pages[i] are copied to the same slots of
 * page dst_pages[i], for every kv head, in both pool arrays (bit exact).
 *
 * This is the copy a prefix cache needs when a new request reuses only the
 * first tokens of a cached page (XY-Serve review, "Assumptions & free
 * parameters": copy-on-write under the block table; Fig. 7, token-wise K/V
 * reuse): the request gets its own page, starting with those tokens' K/V.
 *  src_pages, dst_pages, num_slots  device int32 [count].
 * Enqueued on `stream`; a page id outside [0, num_pages) or a slot count outside
 * [0, page_size] is skipped and recorded in the device error word
 * (PPS_DEV_ERR_COPY_ARGUMENT).  The copies of one call run concurrently: no
 * destination page may also be a source page of the same call (issue them in
 * separate calls, in order, when that happens).
 */
pps_status pps_copy_slots(const pps_pool* pool, const int32_t* src_pages, const int32_t* dst_pages,
                          const int32_t* num_slots, int32_t count, void* stream);

/*
 * Host radix-tree prefix cache with a page allocator (pps_cache_*): the step
 * that produces the page lists pps_kv_append and pps_attn_plan consume.
 *
 * Sources: SGLang review, "Core claim" (RadixAttention: the KV of finished
 * requests stays in a radix tree and later requests sharing a prefix reuse
 * it); XY-Serve review, "Assumptions & free parameters" and Fig. 7 (block
 * table plus radix tree under copy-on-write and eviction; token-wise reuse);
 * attentionhub.org listing, cache-replacement entries (LRU and LFU eviction).
 * The pages fix no algorithm; these rules are the plain reading:
 *  - One tree node is one page of the pool: a chunk of up to page_size token
 *    ids.  A chunk shorter than a page (a finished request's partly filled last
 *    page) is always a leaf.
 *  - pps_cache_begin walks the tree from the root: among the children, the one
 *    whose chunk shares the longest prefix with the next tokens wins (ties: the
 *    lower page id).  A whole full page matched is shared and the walk goes on;
 *    a partly matched page is reused token-wise by copy-on-write into the
 *    request's first new page (out_copy).  At most n - 1 tokens are reused, so
 *    a request always computes its last token.
 *  - Pages are handed out lowest id first.  With none free, one evictable node
 *    (a leaf whose page no active request holds) is evicted and its page reused:
 *    the smallest (last use, page id) with PPS_CACHE_LRU, the smallest (hits,
 *    last use, page id) with PPS_CACHE_LFU.  Every call advances a tick; a
 *    node's last use is the tick of the last call that matched, copied from or
 *    walked it; its hits count the begin calls that reused it.
 *  - pps_cache_finish inserts the request's pages below its matched path: a
 *    chunk equal to an existing child's drops the request's page (freed unless
 *    still held) and follows that child; otherwise the page becomes a new node.
 *  - A call that needs pages when none are free and nothing is evictable
 *    returns PPS_ERR_CACHE_FULL and gives back the pages it took (evictions it
 *    already made stay made); the request is not started or not extended.
 * Typical step: pps_cache_begin / pps_cache_extend per request, pps_copy_slots
 * for the returned copies, pps_kv_append of positions [cached_len, n), then
 * pps_attn_plan with kv_len = n over the pages from pps_cache_request_pages.
 * Enqueue each copy (on one stream) before making the next cache call, and the
 * step's appends before the next step's: a page evicted by a later call can be
 * handed out again at once.  A cache is not thread safe; it holds host memory
 * only.
 */
#define PPS_CACHE_LRU 0
#define PPS_CACHE_LFU 1
typedef struct pps_cache pps_cache;
typedef struct pps_cache_stats {
  int32_t num_pages, page_size, free_pages, active_requests;
  int64_t tree_nodes;      /* pages held by the tree                               */
  int64_t evictions;       /* nodes evicted so far                                 */
  int64_t reused_tokens;   /* sum of cached_len returned by pps_cache_begin         */
  int64_t begun_tokens;    /* sum of n passed to pps_cache_begin                    */
  int64_t tick;            /* calls so far                                         */
} pps_cache_stats;

/* A cache over pool pages [0, num_pages) of page_size slots. */
pps_status pps_cache_create(int32_t num_pages, int32_t page_size, int32_t policy,
                            pps_cache** out_cache);
pps_status pps_cache_destroy(pps_cache* cache);
/* Starts a request of n >= 1 tokens (host int32 ids).  Outputs: its id, the
 * number of leading tokens whose K/V is already in its pages (cached_len), and
 * out_copy[3] = {src page, dst page, slots} (slots 0: no copy needed). */
pps_status pps_cache_begin(pps_cache* cache, const int32_t* tokens, int32_t n,
                           int32_t* out_request, int32_t* out_cached_len, int32_t* out_copy);
/* Appends m tokens (decode); *out_first_position (optional) = their first position. */
pps_status pps_cache_extend(pps_cache* cache, int32_t request, const int32_t* tokens, int32_t m,
                            int32_t* out_first_position);
/* Ends a request; insert != 0 keeps its pages in the tree for reuse. */
pps_status pps_cache_finish(pps_cache* cache, int32_t request, int32_t insert);
/* The request's page list (valid until its next extend or finish). */
pps_status pps_cache_request_pages(const pps_cache* cache, int32_t request,
                                   const int32_t** pages, int32_t* num_pages,
                                   int32_t* num_tokens);
/* pps_cache_extend for many requests in one call: request requests[i] gets
 * tokens [token_indptr[i], token_indptr[i + 1]).  out_first_positions
 * (optional) receives each request's first new position.  Stops at the first
 * failure (PPS_ERR_CACHE_FULL, or an unknown request) with *out_done = the
 * number of requests already extended. */
pps_status pps_cache_extend_batch(pps_cache* cache, const int32_t* requests,
                                  const int32_t* token_indptr, const int32_t* tokens,
                                  int32_t count, int32_t* out_first_positions, int32_t* out_done);
/* The batch's CSR page table for pps_kv_append / pps_attn_plan: kv_len[count]
 * (tokens each request holds), page_indptr[count + 1] and page_indices (room
 * for `capacity` entries), for requests[0..count) in that order. */
pps_status pps_cache_tables(const pps_cache* cache, const int32_t* requests, int32_t count,
                            int32_t* kv_len, int32_t* page_indptr, int32_t* page_indices,
                            int64_t capacity);
pps_status pps_cache_get_stats(const pps_cache* cache, pps_cache_stats* stats);
/* Tree contents for inspection: per node (5 + page_size) int64 values {page,
 * parent's page or -1, chunk length, last use, hits, chunk (padded with -1)}.
 * *needed = values required; with capacity 0 only *needed is set. */
pps_status pps_cache_dump(const pps_cache* cache, int64_t* out, int64_t capacity,
                          int64_t* needed);

/*
 * Host token-wise budget scheduler (pps_sched_*): forms each step's mixed
 * batch from the prefill, decode and verify queues.
 *
 * Sources: XY-Serve review, "Core claim" (a token-wise scheduler selects a
 * budgeted chunk of tokens from mixed prefill, decode and verify queues, with
 * SplitFuse-style chunking) and Fig. 6 (prefills are split so every scheduled
 * chunk stays within the budget; some slots are reserved for decode and
 * speculative tokens to keep the time between tokens stable).  Plain reading:
 *  - A step holds at most `budget` tokens; prefill never uses the last
 *    `reserved` of them.
 *  - Generation requests (decode: 1 token per step; verify: its draft length)
 *    come first, in the order they started generating, each whole; one that
 *    does not fit in what is left waits (later ones may still fit).
 *  - Then prefill requests, first come first served: each takes
 *    min(its remaining prompt tokens, the prefill room left, the step left);
 *    when either runs out the rest wait (chunked prefill).
 *  - A request whose prompt is done starts generating at the next step.
 * The caller feeds each step's batch to the prefix cache and the attention
 * path (q = the tokens the scheduler gave the request) and removes finished
 * requests.  Host memory only; not thread safe.
 */
typedef struct pps_sched pps_sched;
pps_status pps_sched_create(int32_t budget, int32_t reserved, pps_sched** out_sched);
pps_status pps_sched_destroy(pps_sched* sched);
/* Queues a request id (not already queued) with prompt_tokens still to compute
 * (0: it generates from the next step) and gen_tokens >= 1 per generation step. */
pps_status pps_sched_add(pps_sched* sched, int32_t request, int32_t prompt_tokens,
                         int32_t gen_tokens);
pps_status pps_sched_remove(pps_sched* sched, int32_t request);
/* Changes the tokens per generation step (e.g. a new draft length). */
pps_status pps_sched_set_gen_tokens(pps_sched* sched, int32_t request, int32_t gen_tokens);
/* Forms the next batch: entries (request, tokens, is_prefill), generation
 * entries first.  Fails with PPS_ERR_INVALID_ARGUMENT, changing nothing, if it
 * has more than `capacity` entries. */
pps_status pps_sched_step(pps_sched* sched, int32_t* out_requests, int32_t* out_tokens,
                          int32_t* out_is_prefill, int32_t capacity, int32_t* out_count);
pps_status pps_sched_counts(const pps_sched* sched, int32_t* prefill_requests,
                            int64_t* prefill_tokens, int32_t* gen_requests);

/*
 * pps_gemm_bf16 -- the projection GEMM of a mixed batch: C = A W^T.
 *
 * XY-Serve review, "Core claim": SmoothGEMM serves arbitrary shapes with the
 * efficiency of a fixed-shape kernel by padding virtually in on-chip buffers
 * and reading / writing only real data.  Here the fixed shape is a 128 x 256
 * output tile on the tensor cores (tcgen05); a tile that runs past M, N or K is
 * zero-padded in shared memory only, and only rows < M, columns < N are stored.
 *  a  device bf16 [M, K] row-major (token rows; M may be any value >= 0)
 *  w  device bf16 [N, K] row-major (one weight row per output column)
 *  c  device bf16 [M, N] row-major, written (fp32 accumulation, RNE to bf16)
 * N and K must be multiples of 8 (16-byte rows); pointers 16-byte aligned.
 * Enqueued on `stream`.  A pipeline wait that runs out is recorded in the
 * device error word (PPS_DEV_ERR_WAIT_TIMEOUT).
 */
pps_status pps_gemm_bf16(const void* a, const void* w, void* c, int32_t M, int32_t N, int32_t K,
                         void* stream);

/*
 * pps_partition -- split one batch over num_parts GPUs so that no data has to
 * move between them: every radix subtree (the requests whose first whole
 * cached page is the same page, i.e. that share a cached prefix) stays on one
 * GPU, where its shared pages are still read once, and the subtrees are
 * balanced by work.  XY-Serve review, "What carries the argument" (work sorted
 * by area and spread so every core gets a fair share); SGLang review, "Core
 * claim" (prefix reuse).  Rules:
 *  - a request with no whole cached page is a subtree of its own;
 *  - work of a request = max(1, new tokens) x kv_len; of a subtree, the sum;
 *  - subtrees by work, largest first (ties: lowest request id in it), each to
 *    the part with the least work so far (ties: lowest part).
 * Host arrays as in pps_attn_plan; out_part [num_requests] receives the part
 * of each request, out_load [num_parts] (optional) the work of each part.
 * Each GPU then plans and runs its own requests (no collective).
 */
pps_status pps_partition(const int32_t* q_indptr, const int32_t* kv_len,
                         const int32_t* page_indptr, const int32_t* page_indices,
                         int32_t num_requests, int32_t page_size, int32_t num_parts,
                         int32_t* out_part, int64_t* out_load);

/*
 * Serving-step runtime (pps_engine_*): a prefix cache (pps_cache_*) and a
 * token-wise scheduler (pps_sched_*) kept together, so that one step of a
 * serving loop is two native calls instead of a call per request:
 *  1. pps_engine_schedule picks the batch: entries (request, tokens,
 *     is_prefill), generation entries first (pps_sched_step).
 *  2. pps_engine_commit takes the new token ids of the batch's generation
 *     entries (concatenated in batch order: gen_tokens), appends them to the
 *     cache, moves the prefill entries forward, and writes the tables of the
 *     entries it kept, ready for pps_kv_append (cached_len) and pps_attn_plan
 *     (kv_len, page CSR): out_requests[k], q_indptr[k + 1], cached_len[k],
 *     kv_len[k], page_indptr[k + 1], page_indices.  A generation entry the cache
 *     has no page for is left out (the scheduler picks it again next step).
 *     page_capacity (entries of page_indices) must cover every entry's pages
 *     plus 1 + tokens / page_size per generation entry; that bound is written
 *     to *out_pages_needed (may be NULL) and checked before anything changes:
 *     PPS_ERR_INVALID_ARGUMENT if it is short, the batch still pending.
 * pps_engine_add admits a request (pps_cache_begin + pps_sched_add; copy as
 * pps_cache_begin), pps_engine_finish retires one (pps_sched_remove +
 * pps_cache_finish).  Neither may be called between schedule and commit.
 * pps_engine_parts exposes the cache and the scheduler (owned by the engine)
 * for their stats.  Host memory only; not thread safe.
 */
typedef struct pps_engine pps_engine;
pps_status pps_engine_create(int32_t num_pages, int32_t page_size, int32_t cache_policy,
                             int32_t budget, int32_t reserved, pps_engine** out_engine);
pps_status pps_engine_destroy(pps_engine* engine);
pps_status pps_engine_parts(pps_engine* engine, pps_cache** cache, pps_sched** sched);
pps_status pps_engine_add(pps_engine* engine, const int32_t* tokens, int32_t n, int32_t gen_tokens,
                          int32_t* out_request, int32_t* out_cached_len, int32_t* out_copy);
pps_status pps_engine_finish(pps_engine* engine, int32_t request, int32_t insert);
pps_status pps_engine_schedule(pps_engine* engine, int32_t* out_requests, int32_t* out_tokens,
                               int32_t* out_is_prefill, int32_t capacity, int32_t* out_count);
pps_status pps_engine_commit(pps_engine* engine, const int32_t* gen_tokens,
                             int32_t* out_requests, int32_t* q_indptr, int32_t* cached_len,
                             int32_t* kv_len, int32_t* page_indptr, int32_t* page_indices,
                             int64_t page_capacity, int64_t* out_pages_needed,
                             int32_t* out_count);

/* Optional planner knobs; pass NULL for defaults.  Zero fields take defaults. */
typedef struct pps_plan_options {
  int32_t num_sms;          /* SMs to balance over; 0 = query the current device (152 if none) */
  int32_t bw_chunk_tokens;  /* KV tokens per split-KV task on the bandwidth path; 0 = adaptive    */
  int32_t mma_chunk_tokens; /* KV tokens per tensor-core task (multiple of 128); 0 = adaptive     */
  int32_t flags;            /* PPS_PLAN_* bits                                                   */
} pps_plan_options;

#define PPS_PLAN_NO_GROUPS 1      /* do not merge shared-prefix pages into group tasks            */
#define PPS_PLAN_CUDA_CORES_ONLY 2 /* route every task to the CUDA-core kernel (no tcgen05 tiles) */
#define PPS_PLAN_SMALL_ROWS_CUDA_CORES 4 /* tasks of few rows on the CUDA-core kernel, not the key-tile one */
#define PPS_PLAN_FUSED_APPEND 8    /* step calls: the first attention kernel appends the rows (no separate launch) */

typedef struct pps_plan pps_plan;

/*
 * pps_attn_plan -- decompose one batch into a work-sorted tile task table.
 *
 * Host-only (no CUDA call unless opts->num_sms is 0 and a device exists).
 * Follows the XY-Serve review's workload decomposition and task reordering
 * ("Core claim", "What carries the argument"):
 *  1. a radix tree over each request's fully cached page ids finds runs of
 *     pages shared by >= 2 requests (SGLang review, "Core claim"); each run
 *     becomes one group task per kv head that attends all of its members'
 *     query rows against those pages, so shared pages are read once per group;
 *  2. each request's remaining positions (private pages and this step's new
 *     tokens, causal) become request tasks;
 *  3. tasks with few query rows go to the bandwidth (split-KV, CUDA-core)
 *     kernel, wider ones to the tcgen05 tensor-core kernel in 128-row tiles;
 *     fully masked causal tiles are never created;
 *  4. tasks are sorted by work (rows x KV tokens) in descending order;
 *  5. every (token, head) covered by more than one task gets partial slots
 *     that a merge kernel combines by log-sum-exp.
 *
 *  q_indptr     host int32 [num_requests + 1]: new-token offsets (q_indptr[0] = 0).
 *  kv_len       host int32 [num_requests]: cached + new tokens of each request.
 *  page_indptr  host int32 [num_requests + 1]; page_indices host int32 [nnz]
 *               (identical ids in two requests' lists mean shared pages).
 *  num_pages    pool size, for range checks.
 *  sm_scale     softmax scale (normally 1/sqrt(head_dim)); must be finite.
 * On success *out_plan owns a host copy of everything the kernels need and
 * *out_workspace_bytes is the device workspace pps_attn_run requires.
 * The input arrays may be freed or changed after the call returns.
 * Errors: PPS_ERR_INVALID_ARGUMENT, PPS_ERR_UNSUPPORTED, PPS_ERR_PAGE_TABLE,
 * PPS_ERR_NO_MEMORY; *out_plan is then NULL.
 */
pps_status pps_attn_plan(const int32_t* q_indptr, const int32_t* kv_len,
                         const int32_t* page_indptr, const int32_t* page_indices,
                         int32_t num_requests, int32_t num_q_heads, int32_t num_kv_heads,
                         int32_t head_dim, int32_t page_size, int32_t num_pages, float sm_scale,
                         const pps_plan_options* opts, pps_plan** out_plan,
                         size_t* out_workspace_bytes);

/*
 * pps_attn_plan_tree -- pps_attn_plan for batches whose verify rows are draft
 * trees (tree-based speculative decoding).
 *
 * Sources: XY-Serve review, Fig. 8 (tree-based speculative algorithms keep
 * their predictions for several continuations as one tree that the target
 * model verifies in a single pass); attentionhub.org listing, the Medusa
 * entry (several candidate continuations verified at once with tree-based
 * attention).  The pages fix no mask format; this one is the plain reading:
 *
 *  tree_parent  host int32 [num_new_tokens], or NULL (= pps_attn_plan).
 *               Entry q_indptr[r] + j is the index, among request r's new
 *               tokens, of token j's parent, or -1 when token j hangs
 *               directly off the cached context.  A parent precedes its child
 *               (-1 <= parent < j).  New token j (absolute position c_r + j)
 *               then sees every cached position and the new positions of its
 *               ancestors and itself; other draft positions are masked out.
 *               The chain parent = j - 1 is the ordinary causal mask.
 * The draft tokens' K/V rows are appended at positions c_r + j as usual
 * (pps_kv_append); the tree order is the row order.  A request whose parents
 * are not a chain may have at most PPS_TREE_MAX_TOKENS new tokens.
 * Errors: as pps_attn_plan; PPS_ERR_INVALID_ARGUMENT for a parent out of
 * range, PPS_ERR_UNSUPPORTED for a tree request with too many new tokens.
 */
#define PPS_TREE_MAX_TOKENS 64
pps_status pps_attn_plan_tree(const int32_t* q_indptr, const int32_t* kv_len,
                              const int32_t* page_indptr, const int32_t* page_indices,
                              const int32_t* tree_parent, int32_t num_requests,
                              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t page_size, int32_t num_pages, float sm_scale,
                              const pps_plan_options* opts, pps_plan** out_plan,
                              size_t* out_workspace_bytes);

/*
 * pps_attn_run -- the mixed-batch attention.
 *
 * Runs a plan's tile tasks as the XY-Serve review describes the attention of a
 * P/D/V batch ("Core claim": one matmul-softmax-matmul meta-kernel over the
 * task table, mask sparsity skipping invalid tiles; Fig. 10, the cube working
 * on one tile while the vector unit runs the softmax of another), with the
 * KV split into pieces whose partial softmaxes are merged exactly
 * ("Assumptions & free parameters": online softmax with rescaling equals the
 * plain softmax) and shared-prefix pages read once per group (SGLang review,
 * "Core claim", RadixAttention).
 *
 *  q          device bf16 [num_new_tokens, num_q_heads, head_dim].
 *  pool       host descriptor; its pages must already hold every row the step
 *             attends to (call pps_kv_append first for this step's rows).
 *  out        device bf16 [num_new_tokens, num_q_heads, head_dim]; every row is
 *             written.
 *  workspace  device, >= the plan's workspace bytes, 256-byte aligned; holds the
 *             uploaded task table and fp32 partials.  It must not be used by
 *             other work in flight on another stream.
 * Enqueues: one host-to-device copy of the task table (from the plan's
 * page-locked host memory when a device is usable, so the call does not wait
 * for earlier work), then up to three kernels (bandwidth tasks, tensor-core
 * tasks, partial merge).  The plan may be destroyed as soon as the call
 * returns: the library keeps the table's host memory until the upload has
 * completed.  A plan may be run any number of times.
 * The page-locked table buffers (plans, and the tables of pps_attn_step and
 * pps_attn_step_host) come from a small library pool, each buffer reused once
 * its last upload has completed.  When four buffers large enough for a request
 * are still waiting for their uploads, pps_attn_plan and the step calls wait
 * for the oldest instead of pinning more memory: the host runs at most a few
 * steps ahead of the device.
 */
pps_status pps_attn_run(const pps_plan* plan, const void* q, const pps_pool* pool, void* out,
                        void* workspace, size_t workspace_bytes, void* stream);

/* Same as pps_attn_run, and records caller-created CUDA events (cudaEvent_t
 * passed as void*, any may be NULL) immediately before and after each kernel
 * class: events[2*i] / events[2*i+1] for i = PPS_KERNEL_*.  A class that has
 * no work this step records both events back to back. */
#define PPS_KERNEL_BANDWIDTH 0
#define PPS_KERNEL_TENSOR 1
#define PPS_KERNEL_MERGE 2
#define PPS_NUM_KERNEL_CLASSES 3
pps_status pps_attn_run_events(const pps_plan* plan, const void* q, const pps_pool* pool,
                               void* out, void* workspace, size_t workspace_bytes, void* stream,
                               void* const* events);

/*
 * pps_attn_run_noalloc -- pps_attn_run for callers that cannot allocate device
 * memory.  The paper has no counterpart; this is an integration aid.
 *
 * Some callers cannot call cudaMalloc: a plugin inside an engine that owns all
 * device memory and offers no workspace, or a latency-critical loop that must
 * not reach cudaMalloc / cudaFree (they can synchronize the device).  This call
 * takes the same plan, q, pool and out as pps_attn_run, but instead of a
 * caller workspace it uses a fixed array of PPS_NOALLOC_SCRATCH_BYTES that the
 * library keeps in device memory (every GPU that loads the library holds that
 * array until the process exits).  It allocates nothing.
 *
 *  - A plan whose workspace_bytes exceeds PPS_NOALLOC_SCRATCH_BYTES is
 *    rejected with PPS_ERR_SCRATCH_LIMIT before anything is enqueued.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - All calls share the one array.  It keeps the previous call's contents;
 *    nothing in it needs to start at zero.  Calls whose work overlaps on the
 *    GPU (different streams, or different host threads) race on the array:
 *    order them on one stream or synchronize between them.
 */
#define PPS_NOALLOC_SCRATCH_BYTES (32u << 20)
pps_status pps_attn_run_noalloc(const pps_plan* plan, const void* q, const pps_pool* pool,
                                void* out, void* stream);

/* Frees a plan (host memory only).  NULL is accepted. */
pps_status pps_plan_destroy(pps_plan* plan);

/* Plan summary, for tests and reports. */
typedef struct pps_plan_info {
  int32_t num_requests, num_tokens, num_q_heads, num_kv_heads, head_dim, page_size;
  int32_t num_groups;          /* shared-prefix group nodes found                       */
  int64_t num_bw_tasks;        /* bandwidth-kernel tasks (all kv heads)                 */
  int64_t num_mma_tasks;       /* tensor-core tasks (all kv heads)                      */
  int64_t num_partials;        /* partial slots (per token; x num_q_heads rows each)    */
  int64_t num_merge_tokens;    /* tokens whose rows are combined by the merge kernel    */
  int64_t table_bytes;         /* bytes of the device task table                        */
  int64_t workspace_bytes;
  int64_t kv_bytes_unique;     /* K+V bytes of distinct (page, kv head, valid slot)      */
  int64_t kv_bytes_read;       /* K+V bytes the tasks read (shared runs counted once)    */
  double flops_mma;            /* 4*d per visible (query row, key) pair on tensor tasks  */
  double flops_total;          /* same over all tasks                                   */
  int64_t kv_bytes_bw;         /* K+V bytes the bandwidth tasks read (each once)         */
  double flops_mma_issued;     /* FLOP the tensor core executes: whole 128-row x 128-key tiles */
  int32_t num_tree_requests;   /* requests whose draft is a tree (not a chain)           */
  int32_t small_rows_on_tensor; /* 1: the small-row (bandwidth) tasks run on the key-tile
                                   tcgen05 kernel; 0: on the CUDA-core kernel              */
} pps_plan_info;
pps_status pps_plan_get_info(const pps_plan* plan, pps_plan_info* info);

/*
 * Read-only views of the plan's tables (host memory owned by the plan, valid
 * until pps_plan_destroy).  Task records are PPS_TASK_INTS int32 each:
 *   [0] row_off    first entry of this task's tokens in the ROWS array
 *   [1] n_tok      number of query tokens (rows = n_tok * G)
 *   [2] kv_head
 *   [3] page_off   offset of the request's page list in the PAGES array
 *   [4] kv_begin   first logical KV position read
 *   [5] kv_end     one past the last logical KV position read
 *   [6] causal     token i of the task sees positions <= causal + i
 *                  (PPS_NO_CAUSAL: no causal limit inside [kv_begin, kv_end))
 *   [7] out_pid    -1: write final output rows; else token i writes partial
 *                  slot out_pid + i (rows (out_pid + i) * num_q_heads + h)
 * MERGE_INDPTR / MERGE_PIDS list, for each token in MERGE_TOKENS, its partials.
 * TREE_MASK (plans made with a draft tree only; count 0 otherwise) holds one
 * 64-bit word per new token, as int32 pairs (low word first): bit k is set
 * when the key k positions before the token's own position is visible to it
 * (keys 64 or more positions back are always visible).  Chain tokens hold
 * all ones.  Tasks apply it only when their causal field is not PPS_NO_CAUSAL.
 * TT_CTA (plans whose small-row tasks run on the key-tile tensor kernel only;
 * count 0 otherwise) holds C + 1 offsets for that kernel's C persistent CTAs:
 * CTA b runs BW_TASKS records [TT_CTA[b], TT_CTA[b + 1]) in order.  The
 * planner fills the ranges longest task first, each task to a CTA with the
 * least work so far (whole 128-key tiles plus two per task; ties to the CTA
 * that reached that load first), so within a range the tasks keep descending
 * work; C = min(tasks, SMs).
 * Without TT_CTA, BW_TASKS is in descending work order and persistent CTA b of
 * C takes records b, 2C-1-b, 2C+b, ... (the tensor-core and CUDA-core kernels).
 */
#define PPS_TASK_INTS 8
#define PPS_NO_CAUSAL 0x3fffffff
#define PPS_ARRAY_BW_TASKS 0
#define PPS_ARRAY_MMA_TASKS 1
#define PPS_ARRAY_ROWS 2
#define PPS_ARRAY_PAGES 3
#define PPS_ARRAY_MERGE_TOKENS 4
#define PPS_ARRAY_MERGE_INDPTR 5
#define PPS_ARRAY_MERGE_PIDS 6
#define PPS_ARRAY_TREE_MASK 7
#define PPS_ARRAY_TT_CTA 8
pps_status pps_plan_get_array(const pps_plan* plan, int32_t which, const int32_t** data,
                              int64_t* count);

/*
 * pps_attn_step -- one whole step with the rows already on the device and the
 * tables on the host: the tables are uploaded (through a page-locked staging
 * buffer) into d_scratch, the new K/V rows appended (the pps_kv_append
 * scatter, each new token's page and slot taken on the host from the tables
 * the plan has checked), the batch planned (pps_attn_plan_tree) and attended
 * (pps_attn_run, or pps_attn_run_events when `events` is not NULL).  The same
 * operations as the three device-side calls, in one native call per step.
 *
 *  q, k_new, v_new, out  device bf16 rows as for pps_kv_append / pps_attn_run.
 *  host tables, scratch, errors: as pps_attn_step_host (its scratch holds only
 *  the tables and the plan's workspace here).
 *
 * With opts->flags & PPS_PLAN_FUSED_APPEND (this call and pps_attn_step_host)
 * the append is not a launch of its own: the step's first attention kernel
 * copies the rows into their pages in its set-up, every CTA taking a share,
 * and all its CTAs wait for one another on a counter in the scratch before
 * any reads the pool (XY-Serve review, "Core claim": the step's batch through
 * one meta-kernel; the copy is the pps_kv_append definition, bit exact).  That
 * kernel is launched cooperatively, so all its CTAs are resident at once; the
 * wait is bounded, and one that runs out is recorded as
 * PPS_DEV_ERR_WAIT_TIMEOUT.  It applies when the first kernel is the key-tile
 * kernel (head_dim 128 small-row tasks) or the tensor-core kernel alone; other
 * plans append with a separate launch as without the flag.
 */
pps_status pps_attn_step(const pps_pool* pool, const void* q, const void* k_new, const void* v_new,
                         const int32_t* h_q_indptr, const int32_t* h_kv_len,
                         const int32_t* h_page_indptr, const int32_t* h_page_indices,
                         const int32_t* h_tree_parent, int32_t num_requests, int32_t num_q_heads,
                         float sm_scale, const pps_plan_options* opts, void* out, void* d_scratch,
                         size_t scratch_bytes, size_t* out_scratch_bytes, void* stream,
                         void* const* events);

/*
 * pps_attn_step_host -- one whole step from host memory: the step's new K/V
 * rows, query rows and tables are copied to device scratch, the K/V rows are
 * appended to the pool (as in pps_attn_step), the batch is planned (pps_attn_plan_tree
 * on the host tables) and attended (pps_attn_run), and the output rows are
 * copied back.  The same operations as the device-side calls, in one native
 * call, for a caller that keeps its batch on the host (the XY-Serve review's
 * serving step, "Core claim": each step's mixed batch through one attention).
 *
 *  pool                  host pointer to the pool descriptor (k, v device).
 *  h_q                   host bf16 [T, num_q_heads, head_dim], T = h_q_indptr[R].
 *  h_k_new, h_v_new      host bf16 [T, num_kv_heads, head_dim].
 *  h_q_indptr, h_kv_len, h_page_indptr, h_page_indices, h_tree_parent
 *                        host int32 tables as for pps_attn_plan_tree (tree may be
 *                        NULL); each request's new tokens are its last q_len
 *                        positions (cached_len = kv_len - q_len).
 *  h_out                 host bf16 [T, num_q_heads, head_dim], written when the
 *                        stream reaches the end of this step.  When h_out is
 *                        page-locked memory mapped for the device
 *                        (cudaHostAlloc / cudaHostRegister) and tensor-core
 *                        tiles write at most half of the rows, the step's
 *                        kernels write it directly and no copy follows them;
 *                        otherwise the rows come back by copies after the
 *                        kernels.  When h_out is page-locked, the output
 *                        exceeds 16 MB and comes from two or more requests,
 *                        all on tensor-core tasks with no partials, the tasks
 *                        of the requests holding the first three quarters of
 *                        the tokens run in a launch of their own and their
 *                        rows travel back (on a stream of the library's own)
 *                        while the rest are computed; `stream` waits for that
 *                        copy at the end of the step.
 *  d_scratch             device, 256-byte aligned, scratch_bytes long; the size
 *                        it needs is written to *out_scratch_bytes (may be NULL).
 *                        It holds two slots of input rows taken in turn, room
 *                        for the output rows, the tables and the plan's workspace; it
 *                        must not be used by other work while steps are in
 *                        flight, and steps that share it are issued on one
 *                        stream (steps on other streams take scratch of their own).
 * The copies of the input rows run on a stream of the library's own (one per
 * scratch buffer, up to 32 kept; the least recently used one is retired,
 * after the work it fences has finished, when a 33rd scratch comes), so that
 * the rows of the next call travel while this call's kernels run; the step's
 * kernels on `stream` wait for them, and a slot is written again only once
 * the kernels that read it have finished.  The rest (table upload, append,
 * attention, any output copy) is enqueued on `stream`.
 * Page-locked host rows make the copies asynchronous, and every host buffer
 * must stay valid until the stream has passed this step.  The host tables are
 * read before the call returns.
 * The row copies start before the host plans, so on PPS_ERR_WORKSPACE (scratch
 * missing, misaligned or smaller than needed) or a planning error only the
 * scratch may have been written; the pool is untouched.
 * Errors: as pps_attn_plan_tree and pps_attn_run, and PPS_ERR_WORKSPACE.
 */
pps_status pps_attn_step_host(const pps_pool* pool, const void* h_q, const void* h_k_new,
                              const void* h_v_new, const int32_t* h_q_indptr,
                              const int32_t* h_kv_len, const int32_t* h_page_indptr,
                              const int32_t* h_page_indices, const int32_t* h_tree_parent,
                              int32_t num_requests, int32_t num_q_heads, float sm_scale,
                              const pps_plan_options* opts, void* h_out, void* d_scratch,
                              size_t scratch_bytes, size_t* out_scratch_bytes, void* stream);

/* Reads the current device's error word into *code (0 = none); if `clear`
 * is nonzero, resets it to 0.  Synchronous (waits for the device).  Work on a
 * stream with its own error word (pps_set_stream_error_word) does not touch
 * this one. */
pps_status pps_get_device_error(int32_t* code, int32_t clear);

/*
 * Stream-scoped device error words.  Batches that run concurrently on
 * different streams each need to know whether their own work failed (the
 * XY-Serve review, "Assumptions & free parameters", keeps the block table
 * consistent across requests; an error has to be traced to the batch whose
 * tables caused it).  pps_set_stream_error_word registers a caller-owned
 * device int32 (4-byte aligned, set to 0 by the caller before use) for
 * `stream` on the current device: every later call that enqueues kernels on
 * that stream (pps_kv_append, pps_copy_slots, the attention and step calls,
 * pps_gemm_bf16) records its device-side errors (PPS_DEV_ERR_*) there, the
 * first error of a run of calls winning, instead of in the device's word.
 * d_word NULL removes the registration.  The word must stay valid while work
 * that uses it is in flight; the library never frees it.
 * pps_get_stream_error enqueues a read of the word on `stream` (and, if
 * `clear` is nonzero, a reset to 0 behind it) and waits for the stream:
 * *code = the stream's word, or the device's word when none is registered.
 */
pps_status pps_set_stream_error_word(void* stream, int32_t* d_word);
pps_status pps_get_stream_error(void* stream, int32_t* code, int32_t clear);

/*
 * pps_selftest_wait_timeout -- diagnostic for the kernels' bounded waits.
 * Launches one CTA that waits on a shared-memory mbarrier that nothing ever
 * arrives at, with the same bounded wait the pipelined kernels use, limited to
 * `limit_ns` nanoseconds (clamped to [1 us, 1 s]).  When the limit runs out the
 * kernel records PPS_DEV_ERR_WAIT_TIMEOUT in the device error word and returns;
 * the context stays usable.  No counterpart on the pages (a test hook for the
 * failure path).
 */
pps_status pps_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t pps_launch_count(void);

/* Static description of a status code (never NULL). */
const char* pps_status_string(pps_status status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int32_t pps_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PPS_H_ */
