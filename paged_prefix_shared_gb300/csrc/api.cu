// C ABI of libpps.so (declared in include/pps.h): argument checks, task-table
// upload and kernel launches.  Every step of the attention path runs in this
// library's kernels; there is no host fallback.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "pps_internal.h"
#include "sm100_ptx.cuh"

// Device error word (one per device that loads the library).
__device__ int32_t g_pps_device_error = 0;

namespace {

std::atomic<uint64_t> g_launches{0};

constexpr int kMaxDevices = 64;
int32_t* g_err_ptr[kMaxDevices] = {nullptr};
std::mutex g_err_mu;

// Caller-owned error words registered for streams (pps_set_stream_error_word).
struct StreamWord {
  void* stream;
  int dev;
  int32_t* word;
};
std::vector<StreamWord> g_stream_words;

// The error word for work enqueued on `stream` of the current device: the
// caller's word registered for that stream, else the device's own word
// (looked up once per device).
int32_t* error_word(cudaError_t* status, void* stream) {
  int dev = 0;
  *status = cudaGetDevice(&dev);
  if (*status != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_err_mu);
  for (const StreamWord& w : g_stream_words)
    if (w.stream == stream && w.dev == dev) return w.word;
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    *status = cudaGetSymbolAddress(&p, g_pps_device_error);
    if (*status != cudaSuccess) return nullptr;
    g_err_ptr[dev] = (int32_t*)p;
  }
  return g_err_ptr[dev];
}

bool pool_ok(const pps_pool* p) {
  return p && p->k && p->v && p->num_pages > 0 && p->num_kv_heads > 0 &&
         (p->page_size == 16 || p->page_size == 32 || p->page_size == 64 || p->page_size == 128) &&
         (p->head_dim == 64 || p->head_dim == 128);
}

// What run_impl enqueues: the task-table upload, the kernels, or both (the
// step calls upload before the append, so that the attention kernels follow
// the append kernel directly and may start while it finishes).
enum RunPhase { kRunAll, kRunUpload, kRunKernels };

// Whether the plan's first attention kernel can carry the step's append
// (the key-tile kernel, or the tensor-core kernel when it runs alone).
bool can_fuse_append(const pps_plan* plan) {
  return plan->num_tokens > 0 &&
         ((plan->num_bw > 0 && plan->shape.small_tt) || (plan->num_bw == 0 && plan->num_mma > 0));
}

pps_status run_impl(const pps_plan* plan, const void* q, const pps_pool* pool, void* out,
                    void* workspace, size_t workspace_bytes, void* stream, void* const* events,
                    RunPhase phase = kRunAll, const pps::AppendArgs* app = nullptr,
                    cudaEvent_t split_done = nullptr) {
  if (!plan || !pool || (plan->num_tokens > 0 && (!q || !out))) return PPS_ERR_INVALID_ARGUMENT;
  if (!pool_ok(pool)) return pool && (pool->head_dim != 64 && pool->head_dim != 128) ?
                                  PPS_ERR_UNSUPPORTED : PPS_ERR_INVALID_ARGUMENT;
  const pps::Shape& s = plan->shape;
  if (pool->num_kv_heads != s.num_kv_heads || pool->page_size != s.page_size ||
      pool->head_dim != s.head_dim || pool->num_pages < s.num_pages)
    return PPS_ERR_INVALID_ARGUMENT;
  if (!workspace || workspace_bytes < plan->workspace_bytes || ((uintptr_t)workspace & 255))
    return PPS_ERR_WORKSPACE;
  if (((uintptr_t)q & 15) || ((uintptr_t)out & 15) || ((uintptr_t)pool->k & 15) ||
      ((uintptr_t)pool->v & 15))
    return PPS_ERR_INVALID_ARGUMENT;
  cudaError_t e;
  int32_t* err = error_word(&e, stream);
  if (!err) return PPS_ERR_CUDA;
  auto st = (cudaStream_t)stream;
  auto rec = [&](int i) {
    if (events && events[i]) return cudaEventRecord((cudaEvent_t)events[i], st);
    return cudaSuccess;
  };
  if (plan->num_tokens == 0) {
    if (phase != kRunUpload)
      for (int i = 0; i < 2 * PPS_NUM_KERNEL_CLASSES; ++i)
        if (rec(i) != cudaSuccess) return PPS_ERR_CUDA;
    return PPS_OK;
  }
  char* ws = (char*)workspace;
  if (phase != kRunKernels) {
    // Asynchronous when the plan's table is page-locked; the buffer is not
    // reused before this upload completes, so the plan may be destroyed at once.
    e = cudaMemcpyAsync(ws, plan->image.data, (size_t)plan->image_ints * 4, cudaMemcpyHostToDevice,
                        st);
    if (e != cudaSuccess) return PPS_ERR_CUDA;
    if (pps::host_buf_mark_use(plan->image, stream) != 0) return PPS_ERR_CUDA;
    if (phase == kRunUpload) return PPS_OK;
  }
  const int32_t* base = (const int32_t*)ws;
  const auto& L = plan->layout;
  pps::DeviceTables t;
  t.bw_tasks = (const pps::Task*)(base + L.bw_tasks);
  t.mma_tasks = (const pps::Task*)(base + L.mma_tasks);
  t.rows = base + L.rows;
  t.pages = base + L.pages;
  t.merge_tokens = base + L.merge_tokens;
  t.merge_indptr = base + L.merge_indptr;
  t.merge_pids = base + L.merge_pids;
  t.tree_mask = plan->has_tree ? (const unsigned long long*)(base + L.tree_mask) : nullptr;
  t.tt_cta = plan->shape.tt_ctas > 0 ? base + L.tt_cta : nullptr;
  t.o_part = (float*)(ws + plan->table_bytes);
  t.lse_part = (float*)(ws + plan->table_bytes + plan->partial_o_bytes);
  t.sync = (int32_t*)(ws) + L.sync;

  if (rec(2 * PPS_KERNEL_BANDWIDTH) != cudaSuccess) return PPS_ERR_CUDA;
  if (pps::launch_bw_attention(s, t, plan->num_bw, q, *pool, out, err, stream,
                               plan->num_bw > 0 ? app : nullptr))
    return PPS_ERR_CUDA;
  if (rec(2 * PPS_KERNEL_BANDWIDTH + 1) != cudaSuccess) return PPS_ERR_CUDA;
  if (rec(2 * PPS_KERNEL_TENSOR) != cudaSuccess) return PPS_ERR_CUDA;
  if (split_done && plan->num_mma_first > 0 && !app) {
    // output split: the tasks of the first requests, then (with `split_done`
    // recorded between) the rest, so the first rows can leave while the
    // rest are computed
    pps::DeviceTables t2 = t;
    t2.mma_tasks = t.mma_tasks + plan->num_mma_first;
    if (pps::launch_mma_attention(s, t, plan->num_mma_first, q, *pool, out, err, stream,
                                  nullptr) ||
        cudaEventRecord(split_done, st) != cudaSuccess ||
        pps::launch_mma_attention(s, t2, plan->num_mma - plan->num_mma_first, q, *pool, out, err,
                                  stream, nullptr))
      return PPS_ERR_CUDA;
  } else if (plan->num_mma &&
             pps::launch_mma_attention(s, t, plan->num_mma, q, *pool, out, err, stream,
                                       plan->num_bw == 0 ? app : nullptr)) {
    return PPS_ERR_CUDA;
  }
  if (rec(2 * PPS_KERNEL_TENSOR + 1) != cudaSuccess) return PPS_ERR_CUDA;
  if (rec(2 * PPS_KERNEL_MERGE) != cudaSuccess) return PPS_ERR_CUDA;
  if (pps::launch_merge(s, t, plan->num_merge_tokens, out, stream)) return PPS_ERR_CUDA;
  if (rec(2 * PPS_KERNEL_MERGE + 1) != cudaSuccess) return PPS_ERR_CUDA;
  return PPS_OK;
}

// One thread waits on an mbarrier that never completes; the bounded wait gives
// up after `limit_ns` and the kernel reports it.
__global__ void wait_timeout_selftest_kernel(int32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    sm100::mbar_init(sm100::smem_u32(&bar), 1);
    sm100::fence_mbar_init();
    if (!sm100::mbar_wait(sm100::smem_u32(&bar), 0, limit_ns))
      atomicCAS(err, 0, PPS_DEV_ERR_WAIT_TIMEOUT);
  }
}

}  // namespace

namespace pps {

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// ---- host staging buffers for plan tables -------------------------------------------
// A slot is reused once the upload recorded on it has completed.  A caller
// that enqueues steps faster than the GPU runs them would otherwise pin a new
// buffer every step (and scan an ever longer list); after kRunAhead busy
// slots large enough for a request, the request waits for the oldest upload
// among them instead, so the host runs at most that many steps ahead.
namespace {
constexpr int kRunAhead = 4;
struct HostSlot {
  int32_t* p = nullptr;
  size_t ints = 0;
  bool pinned = false;
  bool in_use = false;
  cudaEvent_t ev = nullptr;   // last upload recorded on this buffer
  int ev_dev = -1;
  uint64_t seq = 0;           // order of that upload
};
std::mutex g_host_mu;
std::vector<HostSlot> g_host;
uint64_t g_host_seq = 0;

bool slot_idle(HostSlot& s) {
  if (!s.ev) return true;
  const cudaError_t q = cudaEventQuery(s.ev);
  if (q == cudaErrorNotReady) return false;
  if (q != cudaSuccess) cudaGetLastError();   // a failed context: the upload is over either way
  return true;
}
}  // namespace

HostBuf host_buf_acquire(size_t ints) {
  std::unique_lock<std::mutex> lk(g_host_mu);
  int best = -1, oldest = -1, busy = 0;
  for (int i = 0; i < (int)g_host.size(); ++i) {
    HostSlot& s = g_host[i];
    if (s.in_use || s.ints < ints) continue;
    if (!slot_idle(s)) {
      ++busy;
      if (oldest < 0 || s.seq < g_host[oldest].seq) oldest = i;
      continue;
    }
    if (best < 0 || s.ints < g_host[best].ints) best = i;
  }
  if (best < 0 && busy >= kRunAhead) {
    // wait for the oldest upload outside the lock; the slot is ours meanwhile
    HostSlot& s = g_host[oldest];
    s.in_use = true;
    const HostBuf b{s.p, s.ints, oldest};
    const cudaEvent_t ev = s.ev;
    lk.unlock();
    if (cudaEventSynchronize(ev) != cudaSuccess) cudaGetLastError();
    return b;
  }
  if (best < 0) {
    size_t cap = 1 << 14;                      // ints; power-of-two classes from 64 KB
    while (cap < ints) cap <<= 1;
    HostSlot s;
    void* p = nullptr;
    if (cudaHostAlloc(&p, cap * 4, cudaHostAllocPortable) == cudaSuccess && p) {
      s.pinned = true;
    } else {
      cudaGetLastError();
      p = std::malloc(cap * 4);
      if (!p) return HostBuf{};
    }
    s.p = (int32_t*)p;
    s.ints = cap;
    g_host.push_back(s);
    best = (int)g_host.size() - 1;
  }
  g_host[best].in_use = true;
  return HostBuf{g_host[best].p, g_host[best].ints, best};
}

void host_buf_release(HostBuf& b) {
  if (b.slot < 0) return;
  std::lock_guard<std::mutex> lk(g_host_mu);
  if (b.slot < (int)g_host.size()) g_host[b.slot].in_use = false;
  b = HostBuf{};
}

int host_buf_mark_use(const HostBuf& b, void* stream) {
  if (b.slot < 0) return 0;
  std::lock_guard<std::mutex> lk(g_host_mu);
  HostSlot& s = g_host[b.slot];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (s.ev && s.ev_dev != dev) {
    cudaEventDestroy(s.ev);
    s.ev = nullptr;
  }
  if (!s.ev) {
    if (cudaEventCreateWithFlags(&s.ev, cudaEventDisableTiming) != cudaSuccess) return 1;
    s.ev_dev = dev;
  }
  s.seq = ++g_host_seq;
  return cudaEventRecord(s.ev, (cudaStream_t)stream) == cudaSuccess ? 0 : 1;
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return 0; }
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace pps

extern "C" {

pps_status pps_kv_append(const pps_pool* pool, const void* k_new, const void* v_new,
                         const int32_t* q_indptr, const int32_t* cached_len,
                         const int32_t* page_indptr, const int32_t* page_indices,
                         int32_t num_requests, int32_t num_new_tokens, void* stream) {
  if (!pool || num_requests < 0 || num_new_tokens < 0) return PPS_ERR_INVALID_ARGUMENT;
  if (pool->head_dim != 64 && pool->head_dim != 128) return PPS_ERR_UNSUPPORTED;
  if (!pool_ok(pool)) return PPS_ERR_INVALID_ARGUMENT;
  if (num_new_tokens == 0) return PPS_OK;
  if (num_requests == 0 || !k_new || !v_new || !q_indptr || !cached_len || !page_indptr ||
      !page_indices)
    return PPS_ERR_INVALID_ARGUMENT;
  if (((uintptr_t)k_new & 15) || ((uintptr_t)v_new & 15) || ((uintptr_t)pool->k & 15) ||
      ((uintptr_t)pool->v & 15))
    return PPS_ERR_INVALID_ARGUMENT;
  cudaError_t e;
  int32_t* err = error_word(&e, stream);
  if (!err) return PPS_ERR_CUDA;
  return pps::launch_kv_append(*pool, k_new, v_new, q_indptr, cached_len, page_indptr,
                               page_indices, num_requests, num_new_tokens, err, stream)
             ? PPS_ERR_CUDA : PPS_OK;
}

pps_status pps_copy_slots(const pps_pool* pool, const int32_t* src_pages, const int32_t* dst_pages,
                          const int32_t* num_slots, int32_t count, void* stream) {
  if (!pool || count < 0) return PPS_ERR_INVALID_ARGUMENT;
  if (pool->head_dim != 64 && pool->head_dim != 128) return PPS_ERR_UNSUPPORTED;
  if (!pool_ok(pool)) return PPS_ERR_INVALID_ARGUMENT;
  if (count == 0) return PPS_OK;
  if (!src_pages || !dst_pages || !num_slots || ((uintptr_t)pool->k & 15) ||
      ((uintptr_t)pool->v & 15))
    return PPS_ERR_INVALID_ARGUMENT;
  cudaError_t e;
  int32_t* err = error_word(&e, stream);
  if (!err) return PPS_ERR_CUDA;
  return pps::launch_copy_slots(*pool, src_pages, dst_pages, num_slots, count, err, stream)
             ? PPS_ERR_CUDA : PPS_OK;
}

pps_status pps_gemm_bf16(const void* a, const void* w, void* c, int32_t M, int32_t N, int32_t K,
                         void* stream) {
  if (M < 0 || N <= 0 || K <= 0 || (N % 8) || (K % 8)) return PPS_ERR_INVALID_ARGUMENT;
  if (M == 0) return PPS_OK;
  if (!a || !w || !c || ((uintptr_t)a & 15) || ((uintptr_t)w & 15) || ((uintptr_t)c & 15))
    return PPS_ERR_INVALID_ARGUMENT;
  cudaError_t e;
  int32_t* err = error_word(&e, stream);
  if (!err) return PPS_ERR_CUDA;
  return pps::launch_gemm_bf16(a, w, c, M, N, K, err, stream) ? PPS_ERR_CUDA : PPS_OK;
}

pps_status pps_attn_run(const pps_plan* plan, const void* q, const pps_pool* pool, void* out,
                        void* workspace, size_t workspace_bytes, void* stream) {
  return run_impl(plan, q, pool, out, workspace, workspace_bytes, stream, nullptr);
}

pps_status pps_attn_run_events(const pps_plan* plan, const void* q, const pps_pool* pool,
                               void* out, void* workspace, size_t workspace_bytes, void* stream,
                               void* const* events) {
  return run_impl(plan, q, pool, out, workspace, workspace_bytes, stream, events);
}

}  // extern "C"

namespace {

// The host-to-device row copies of pps_attn_step_host run on a stream of the
// library's own, into one of two row slots of the scratch taken in turn, so
// the next step's rows travel while this step's kernels run.  A slot is
// written again only after the kernels that read it (event `free`), and the
// step's kernels wait for their slot's copies (event `in`).  The state is kept
// per scratch buffer (device, address), so steps on several streams, each with
// its own scratch, never wait on one another's events.
struct RowCopier {
  int dev = -1;
  const void* scratch = nullptr;
  uint64_t last_use = 0;
  cudaStream_t copy = nullptr;
  cudaEvent_t in[2] = {nullptr, nullptr};
  cudaEvent_t free[2] = {nullptr, nullptr};
  bool used[2] = {false, false};
  uint64_t calls = 0;
  // output split: the first requests' rows go back on `out` once their
  // tensor-core launch is done (`split`), while the rest are computed
  cudaStream_t out = nullptr;
  cudaEvent_t split = nullptr, out_done = nullptr;
};
constexpr int kMaxCopiers = 32;
std::mutex g_copier_mu;
RowCopier g_copier[kMaxCopiers];
uint64_t g_copier_clock = 0;

// The copier of `scratch` on the current device; a new scratch takes a free
// entry, else the least recently used one once the work it fenced has
// finished.  Null on a CUDA error.  Called with g_copier_mu held.
RowCopier* row_copier(const void* scratch) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  RowCopier* pick = nullptr;
  for (RowCopier& c : g_copier)
    if (c.dev == dev && c.scratch == scratch) { pick = &c; break; }
  if (!pick) {
    for (RowCopier& c : g_copier)
      if (!pick || c.last_use < pick->last_use) pick = &c;
    RowCopier& c = *pick;
    if (c.copy) {
      // the entry's own resources belong to its device; wait for what they fence
      int cur = dev;
      if (cudaSetDevice(c.dev) != cudaSuccess) return nullptr;
      bool ok = cudaStreamSynchronize(c.copy) == cudaSuccess &&
                cudaStreamSynchronize(c.out) == cudaSuccess;
      for (int i = 0; i < 2; ++i) ok = ok && cudaEventSynchronize(c.free[i]) == cudaSuccess;
      cudaStreamDestroy(c.copy);
      cudaStreamDestroy(c.out);
      for (int i = 0; i < 2; ++i) { cudaEventDestroy(c.in[i]); cudaEventDestroy(c.free[i]); }
      cudaEventDestroy(c.split);
      cudaEventDestroy(c.out_done);
      c = RowCopier{};
      if (cudaSetDevice(cur) != cudaSuccess || !ok) return nullptr;
    }
    bool ok = cudaStreamCreateWithFlags(&c.copy, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&c.out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&c.split, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&c.out_done, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; i < 2; ++i)
      ok = ok && cudaEventCreateWithFlags(&c.in[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&c.free[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      if (c.copy) cudaStreamDestroy(c.copy);
      if (c.out) cudaStreamDestroy(c.out);
      if (c.split) cudaEventDestroy(c.split);
      if (c.out_done) cudaEventDestroy(c.out_done);
      for (int i = 0; i < 2; ++i) {
        if (c.in[i]) cudaEventDestroy(c.in[i]);
        if (c.free[i]) cudaEventDestroy(c.free[i]);
      }
      c = RowCopier{};
      return nullptr;
    }
    c.dev = dev;
    c.scratch = scratch;
  }
  pick->last_use = ++g_copier_clock;
  return pick;
}

// The address by which the current device reaches host byte `p`, if `p` lies
// in page-locked host memory mapped for it; else null.
void* device_view_of_host(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();                      // not a CUDA pointer: clear the error
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// One step: rows on the host (copied into scratch first) or already on the
// device; host tables uploaded through a page-locked staging buffer; append,
// plan, attention; rows out (to the host, or left in the caller's device
// output).  The row copies start before the host plans.
pps_status step_impl(const pps_pool* pool, const void* q, const void* k_new, const void* v_new,
                     bool rows_on_host, const int32_t* h_q_indptr, const int32_t* h_kv_len,
                     const int32_t* h_page_indptr, const int32_t* h_page_indices,
                     const int32_t* h_tree_parent, int32_t num_requests, int32_t num_q_heads,
                     float sm_scale, const pps_plan_options* opts, void* out, void* d_scratch,
                     size_t scratch_bytes, size_t* out_scratch_bytes, void* stream,
                     void* const* events) {
  if (out_scratch_bytes) *out_scratch_bytes = 0;
  if (!pool_ok(pool) || num_requests < 0 || num_q_heads <= 0 || !h_q_indptr ||
      (num_requests > 0 && (!h_kv_len || !h_page_indptr)))
    return pool && (pool->head_dim != 64 && pool->head_dim != 128) ? PPS_ERR_UNSUPPORTED
                                                                     : PPS_ERR_INVALID_ARGUMENT;
  const int32_t R = num_requests;
  const int32_t T = h_q_indptr[R];
  if (T < 0 || (T > 0 && (!q || !k_new || !v_new || !out))) return PPS_ERR_INVALID_ARGUMENT;
  // Device scratch: [rows in and out, host rows only] tables, then the plan's
  // workspace.  Everything before the workspace is sized by the batch alone.
  auto al = [](size_t n) { return (n + 255) / 256 * 256; };
  const size_t D = (size_t)pool->head_dim;
  const size_t q_bytes = (size_t)T * num_q_heads * D * 2;
  const size_t kv_bytes = (size_t)T * pool->num_kv_heads * D * 2;
  const int64_t nnz = R > 0 ? h_page_indptr[R] : 0;
  if (nnz < 0 || (nnz > 0 && !h_page_indices)) return PPS_ERR_INVALID_ARGUMENT;
  // tables: q_indptr, cached_len, page_indptr, page_indices, then (8-byte
  // aligned) each new token's {page, slot} for the append
  const size_t slots_off = ((size_t)(R + 1) + R + (R + 1) + (size_t)nnz + 1) & ~(size_t)1;
  const size_t tab_ints = slots_off + 2 * (size_t)T;
  // host rows: two input slots (q, k, v each) and one output area
  const size_t slot_bytes = al(q_bytes) + 2 * al(kv_bytes);
  const size_t rows = rows_on_host ? 2 * slot_bytes + al(q_bytes) : 0;
  const size_t off_k = al(q_bytes), off_v = off_k + al(kv_bytes), off_out = 2 * slot_bytes,
               off_tab = rows, off_ws = off_tab + al(tab_ints * 4);
  // Host rows with a large output from several requests: the planner puts
  // the tensor-core tasks of the requests holding the first three quarters of
  // the tokens first, so those rows can go back to the host while the rest
  // are computed (the device-to-host copy after the kernels is otherwise the
  // one part of a host-row step nothing overlaps; a long-prefill step measured
  // 35.1-35.8 ms with the split at half the tokens, 34.3-35.6 at three
  // quarters, 37.1-38.1 without).  Page-locked output only: a copy into
  // pageable memory would hold the host until the first launch is done.
  auto split_request = [&](bool locked_out) {
    int32_t r1 = 0;
    if (rows_on_host && locked_out && R >= 2 && T > 0 && q_bytes >= ((size_t)16 << 20)) {
      r1 = 1;
      while (r1 < R - 1 && h_q_indptr[r1] < T / 4 * 3) ++r1;
    }
    return r1;
  };
  auto plan_for = [&](pps_plan** pl, size_t* ws, int32_t split_req) {
    return pps::plan_tree(h_q_indptr, h_kv_len, h_page_indptr, h_page_indices, h_tree_parent, R,
                          num_q_heads, pool->num_kv_heads, pool->head_dim, pool->page_size,
                          pool->num_pages, sm_scale, opts, split_req, pl, ws);
  };
  if (!d_scratch || scratch_bytes < off_ws || ((uintptr_t)d_scratch & 255)) {
    // report the whole size (rows, tables and the plan's workspace); nothing enqueued
    pps_plan* probe = nullptr;
    size_t ws = 0;
    const pps_status ps = plan_for(&probe, &ws, 0);
    if (ps != PPS_OK) return ps;
    pps_plan_destroy(probe);
    if (out_scratch_bytes) *out_scratch_bytes = off_ws + al(ws);
    return PPS_ERR_WORKSPACE;
  }
  char* sc = (char*)d_scratch;
  auto stm = (cudaStream_t)stream;
  const void* dq = q;
  const void* dk = k_new;
  const void* dv = v_new;
  void* dout = out;
  RowCopier* rc = nullptr;
  int slot = 0;
  void* host_out = nullptr;
  bool out_direct = false;
  if (rows_on_host) {
    // rows in, on the copier's stream into the next slot (only the scratch is
    // written until the plan is known); the step's kernels wait for them
    std::lock_guard<std::mutex> lk(g_copier_mu);
    rc = row_copier(d_scratch);
    if (!rc) return PPS_ERR_CUDA;
    slot = (int)(rc->calls++ & 1);
    char* sl = sc + slot * slot_bytes;
    if (rc->used[slot] && cudaStreamWaitEvent(rc->copy, rc->free[slot], 0) != cudaSuccess)
      return PPS_ERR_CUDA;
    if (T > 0 &&
        (cudaMemcpyAsync(sl, q, q_bytes, cudaMemcpyHostToDevice, rc->copy) != cudaSuccess ||
         cudaMemcpyAsync(sl + off_k, k_new, kv_bytes, cudaMemcpyHostToDevice, rc->copy) != cudaSuccess ||
         cudaMemcpyAsync(sl + off_v, v_new, kv_bytes, cudaMemcpyHostToDevice, rc->copy) != cudaSuccess))
      return PPS_ERR_CUDA;
    if (cudaEventRecord(rc->in[slot], rc->copy) != cudaSuccess ||
        cudaStreamWaitEvent(stm, rc->in[slot], 0) != cudaSuccess)
      return PPS_ERR_CUDA;
    dq = sl;
    dk = sl + off_k;
    dv = sl + off_v;
    dout = sc + off_out;
    // output rows in page-locked host memory the device can address (first
    // and last byte mapped for this device)?
    if (T > 0) {
      void* d0 = device_view_of_host(out);
      void* d1 = device_view_of_host((const char*)out + q_bytes - 1);
      if (d0 && d1 == (char*)d0 + q_bytes - 1) host_out = d0;
    }
  }
  // the plan, from the host tables (checks them all)
  pps_plan* plan = nullptr;
  size_t ws_bytes = 0;
  pps_status st = plan_for(&plan, &ws_bytes, split_request(host_out != nullptr));
  if (st != PPS_OK) return st;
  const size_t need = off_ws + al(ws_bytes);
  if (out_scratch_bytes) *out_scratch_bytes = need;
  if (scratch_bytes < need) {
    pps_plan_destroy(plan);
    return PPS_ERR_WORKSPACE;
  }
  // Output rows into mapped host memory straight from the kernels, so no
  // copy follows the step -- unless tensor-core tiles write most of them: that
  // kernel's epilogue stalls on stores that cross to host memory (a
  // long-prefill step, all rows on tensor-core tiles, measured 37 -> 41 ms).
  // Those batches, and host memory the device cannot address, get the rows
  // through scratch and a copy on `stream`.
  int64_t mma_rows = 0;
  const int32_t* mt = plan->image.data + plan->layout.mma_tasks;
  for (int64_t i = 0; i < plan->num_mma; ++i) mma_rows += mt[i * PPS_TASK_INTS + 1];
  mma_rows *= plan->shape.group;
  if (host_out && 2 * mma_rows <= (int64_t)T * num_q_heads) {
    dout = host_out;
    out_direct = true;
  }
  // tables (q_indptr, cached_len = kv_len - q_len, page CSR) through one
  // page-locked staging buffer, reused only after this upload completes; for
  // a plan whose task table is small, the task table rides in the same copy
  // (scratch holds them back to back), one copy-engine round trip fewer ahead
  // of the append
  const size_t tab_span = off_ws - off_tab;               // the tables, 256-byte rounded
  const size_t img_bytes = (size_t)plan->image_ints * 4;
  const bool one_copy = T > 0 && img_bytes <= ((size_t)1 << 20);
  const size_t stage_ints = one_copy ? (tab_span + img_bytes) / 4 : tab_ints;
  pps::HostBuf tb = pps::host_buf_acquire(std::max<size_t>(stage_ints, 1));
  if (!tb.data) {
    pps_plan_destroy(plan);
    return PPS_ERR_NO_MEMORY;
  }
  int32_t* t = tb.data;
  std::memcpy(t, h_q_indptr, (size_t)(R + 1) * 4);
  for (int32_t r = 0; r < R; ++r) t[R + 1 + r] = h_kv_len[r] - (h_q_indptr[r + 1] - h_q_indptr[r]);
  if (R > 0) std::memcpy(t + 2 * R + 1, h_page_indptr, (size_t)(R + 1) * 4);
  if (nnz) std::memcpy(t + 3 * R + 2, h_page_indices, (size_t)nnz * 4);
  // every new token's destination; the plan has checked the page lists
  // (long enough for kv_len, ids in range)
  {
    const int32_t P = pool->page_size;
    int32_t* ds = t + slots_off;
    for (int32_t r = 0; r < R; ++r) {
      const int32_t q0 = h_q_indptr[r], c = h_kv_len[r] - (h_q_indptr[r + 1] - q0);
      const int32_t* pl = h_page_indices + h_page_indptr[r];
      for (int32_t j = q0; j < h_q_indptr[r + 1]; ++j) {
        const int32_t pos = c + (j - q0);
        ds[2 * (size_t)j] = pl[pos / P];
        ds[2 * (size_t)j + 1] = pos % P;
      }
    }
    if (slots_off > (size_t)(3 * R + 2) + (size_t)nnz) t[slots_off - 1] = 0;   // the pad word
  }
  if (one_copy) {
    std::memset(t + tab_ints, 0, tab_span - tab_ints * 4);
    std::memcpy(t + tab_span / 4, plan->image.data, img_bytes);
  }
  bool ok = cudaMemcpyAsync(sc + off_tab, t, one_copy ? tab_span + img_bytes : tab_ints * 4,
                            cudaMemcpyHostToDevice, stm) == cudaSuccess;
  ok = ok && pps::host_buf_mark_use(tb, stream) == 0;
  pps::host_buf_release(tb);
  // task table up, append, attend, rows out: the attention kernels directly
  // follow the append kernel, or (PPS_PLAN_FUSED_APPEND) the first of them
  // appends the rows itself
  const int32_t* d_tab = (const int32_t*)(sc + off_tab);
  const bool fused = opts && (opts->flags & PPS_PLAN_FUSED_APPEND) && can_fuse_append(plan);
  const pps::AppendArgs app{dk, dv, d_tab, d_tab + R + 1, d_tab + 2 * R + 1, d_tab + 3 * R + 2,
                            R, T};
  if (ok && !one_copy)
    st = run_impl(plan, dq, pool, dout, sc + off_ws, al(ws_bytes), stream, events, kRunUpload);
  if (ok && st == PPS_OK && !fused && T > 0) {
    if (((uintptr_t)dk & 15) || ((uintptr_t)dv & 15)) st = PPS_ERR_INVALID_ARGUMENT;
    else if (pps::launch_kv_append_slots(*pool, dk, dv, d_tab + slots_off, T, stream))
      st = PPS_ERR_CUDA;
  }
  const bool split_out = rows_on_host && host_out && !out_direct && !fused &&
                         plan->num_mma_first > 0;
  if (ok && st == PPS_OK)
    st = run_impl(plan, dq, pool, dout, sc + off_ws, al(ws_bytes), stream, events, kRunKernels,
                  fused ? &app : nullptr, split_out ? rc->split : nullptr);
  if (rows_on_host) {
    // the slot may be written again once this step's kernels have read it
    std::lock_guard<std::mutex> lk(g_copier_mu);
    if (cudaEventRecord(rc->free[slot], stm) == cudaSuccess) rc->used[slot] = true;
    else ok = false;
  }
  if (ok && st == PPS_OK && rows_on_host && T > 0 && !out_direct) {
    if (split_out) {
      // rows [0, split_tokens) on the copier's output stream once their launch
      // has finished; the stream reaches the end of this step after both copies
      const size_t b1 = (size_t)plan->split_tokens * num_q_heads * D * 2;
      std::lock_guard<std::mutex> lk(g_copier_mu);
      ok = cudaStreamWaitEvent(rc->out, rc->split, 0) == cudaSuccess &&
           cudaMemcpyAsync(out, sc + off_out, b1, cudaMemcpyDeviceToHost, rc->out) ==
               cudaSuccess &&
           cudaEventRecord(rc->out_done, rc->out) == cudaSuccess &&
           cudaMemcpyAsync((char*)out + b1, sc + off_out + b1, q_bytes - b1,
                           cudaMemcpyDeviceToHost, stm) == cudaSuccess &&
           cudaStreamWaitEvent(stm, rc->out_done, 0) == cudaSuccess;
    } else {
      ok = cudaMemcpyAsync(out, sc + off_out, q_bytes, cudaMemcpyDeviceToHost, stm) == cudaSuccess;
    }
  }
  pps_plan_destroy(plan);
  if (!ok) return PPS_ERR_CUDA;
  return st;
}

}  // namespace

extern "C" {

pps_status pps_attn_step_host(const pps_pool* pool, const void* h_q, const void* h_k_new,
                              const void* h_v_new, const int32_t* h_q_indptr,
                              const int32_t* h_kv_len, const int32_t* h_page_indptr,
                              const int32_t* h_page_indices, const int32_t* h_tree_parent,
                              int32_t num_requests, int32_t num_q_heads, float sm_scale,
                              const pps_plan_options* opts, void* h_out, void* d_scratch,
                              size_t scratch_bytes, size_t* out_scratch_bytes, void* stream) {
  return step_impl(pool, h_q, h_k_new, h_v_new, true, h_q_indptr, h_kv_len, h_page_indptr,
                   h_page_indices, h_tree_parent, num_requests, num_q_heads, sm_scale, opts, h_out,
                   d_scratch, scratch_bytes, out_scratch_bytes, stream, nullptr);
}

pps_status pps_attn_step(const pps_pool* pool, const void* q, const void* k_new, const void* v_new,
                         const int32_t* h_q_indptr, const int32_t* h_kv_len,
                         const int32_t* h_page_indptr, const int32_t* h_page_indices,
                         const int32_t* h_tree_parent, int32_t num_requests, int32_t num_q_heads,
                         float sm_scale, const pps_plan_options* opts, void* out, void* d_scratch,
                         size_t scratch_bytes, size_t* out_scratch_bytes, void* stream,
                         void* const* events) {
  if (((uintptr_t)k_new & 15) || ((uintptr_t)v_new & 15)) return PPS_ERR_INVALID_ARGUMENT;
  return step_impl(pool, q, k_new, v_new, false, h_q_indptr, h_kv_len, h_page_indptr,
                   h_page_indices, h_tree_parent, num_requests, num_q_heads, sm_scale, opts, out,
                   d_scratch, scratch_bytes, out_scratch_bytes, stream, events);
}

pps_status pps_get_device_error(int32_t* code, int32_t clear) {
  if (!code) return PPS_ERR_INVALID_ARGUMENT;
  *code = 0;
  if (cudaMemcpyFromSymbol(code, g_pps_device_error, sizeof(int32_t)) != cudaSuccess)
    return PPS_ERR_CUDA;
  if (clear) {
    const int32_t zero = 0;
    if (cudaMemcpyToSymbol(g_pps_device_error, &zero, sizeof(int32_t)) != cudaSuccess)
      return PPS_ERR_CUDA;
  }
  return PPS_OK;
}

pps_status pps_set_stream_error_word(void* stream, int32_t* d_word) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PPS_ERR_CUDA;
  if (d_word && ((uintptr_t)d_word & 3)) return PPS_ERR_INVALID_ARGUMENT;
  std::lock_guard<std::mutex> lk(g_err_mu);
  for (size_t i = 0; i < g_stream_words.size(); ++i)
    if (g_stream_words[i].stream == stream && g_stream_words[i].dev == dev) {
      if (d_word) {
        g_stream_words[i].word = d_word;
      } else {
        g_stream_words.erase(g_stream_words.begin() + (ptrdiff_t)i);
      }
      return PPS_OK;
    }
  if (d_word) g_stream_words.push_back(StreamWord{stream, dev, d_word});
  return PPS_OK;
}

pps_status pps_get_stream_error(void* stream, int32_t* code, int32_t clear) {
  if (!code) return PPS_ERR_INVALID_ARGUMENT;
  *code = 0;
  cudaError_t e;
  int32_t* w = error_word(&e, stream);
  if (!w) return PPS_ERR_CUDA;
  auto st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(code, w, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return PPS_ERR_CUDA;
  if (clear && cudaMemsetAsync(w, 0, sizeof(int32_t), st) != cudaSuccess) return PPS_ERR_CUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? PPS_OK : PPS_ERR_CUDA;
}

pps_status pps_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  if (limit_ns < 1000) limit_ns = 1000;
  if (limit_ns > 1000000000ull) limit_ns = 1000000000ull;
  cudaError_t e;
  int32_t* err = error_word(&e, stream);
  if (!err) return PPS_ERR_CUDA;
  wait_timeout_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(err, limit_ns);
  pps::count_launch();
  return cudaGetLastError() == cudaSuccess ? PPS_OK : PPS_ERR_CUDA;
}

uint64_t pps_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* pps_status_string(pps_status s) {
  switch (s) {
    case PPS_OK: return "ok";
    case PPS_ERR_INVALID_ARGUMENT: return "invalid argument";
    case PPS_ERR_UNSUPPORTED: return "unsupported head_dim, page_size or head ratio";
    case PPS_ERR_PAGE_TABLE: return "malformed page table";
    case PPS_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case PPS_ERR_CUDA: return "CUDA call failed";
    case PPS_ERR_NO_MEMORY: return "host allocation failed";
    case PPS_ERR_SCRATCH_LIMIT: return "plan needs more than the fixed no-alloc scratch";
    case PPS_ERR_CACHE_FULL: return "cache full: no free page and nothing evictable";
    default: return "unknown status";
  }
}

int32_t pps_version(void) { return 220; }

}  // extern "C"
