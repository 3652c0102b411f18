// Internal declarations shared by the host planner, the C ABI and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include "pps.h"

namespace pps {

// One unit of work for one kv head (layout documented in pps.h, PPS_TASK_INTS).
struct Task {
  int32_t row_off;
  int32_t n_tok;
  int32_t kv_head;
  int32_t page_off;
  int32_t kv_begin;
  int32_t kv_end;
  int32_t causal;
  int32_t out_pid;
};
static_assert(sizeof(Task) == PPS_TASK_INTS * 4, "task record size");

// Limits of the kernels.
constexpr int kBwMaxRows = 16;      // query rows (tokens x G) per bandwidth task
constexpr int kMmaRows = 128;       // query rows per tensor-core tile (TMEM lanes)
constexpr int kMmaTaskRows = 256;   // query rows per tensor-core task (two tiles sharing K/V)
constexpr int kMmaKvTile = 128;     // KV positions per tensor-core step
constexpr int kTtRows = 32;         // query rows per key-tile tensor task (head_dim 128)

// Offsets (in int32 units) of the sections of the uploaded task table.
struct TableLayout {
  int64_t bw_tasks = 0, mma_tasks = 0, rows = 0, pages = 0;
  int64_t merge_tokens = 0, merge_indptr = 0, merge_pids = 0;
  int64_t tree_mask = 0;   // 2 ints per new token, only when the plan has a draft tree
  int64_t tt_cta = 0;      // key-tile plans: per-CTA task ranges, CTAs + 1 offsets
  int64_t sync = 0;        // 64 zero ints: the counter of a grid-wide wait
  int64_t total_ints = 0;
};

// Everything the device needs for one run, resolved to device addresses.
struct DeviceTables {
  const Task* bw_tasks;
  const Task* mma_tasks;
  const int32_t* rows;
  const int32_t* pages;
  const int32_t* merge_tokens;
  const int32_t* merge_indptr;
  const int32_t* merge_pids;
  // Per new token, bit k: the key k positions before the token is visible
  // (draft-tree verify); nullptr when the batch has no tree.
  const unsigned long long* tree_mask;
  // Key-tile plans: CTA b runs bw_tasks[tt_cta[b] .. tt_cta[b + 1]).
  const int32_t* tt_cta;
  float* o_part;     // [num_partials, Hq, d]
  float* lse_part;   // [num_partials, Hq] (log2 domain)
  int32_t* sync;     // zero at the start of every run (uploaded with the table)
};

// The step's new K/V rows, appended by the first attention kernel of the
// step itself (the append fused into the attention launch): rows as for
// pps_kv_append, tables on the device.
struct AppendArgs {
  const void* k_new;
  const void* v_new;
  const int32_t* q_indptr;
  const int32_t* cached_len;
  const int32_t* page_indptr;
  const int32_t* page_indices;
  int32_t num_requests;
  int32_t num_tokens;
};

struct Shape {
  int32_t num_q_heads, num_kv_heads, head_dim, page_size, group;  // group = G
  int32_t num_pages;
  float sm_scale;
  int32_t bw_rows_max;   // largest n_tok * G over bandwidth tasks
  int32_t small_tt;      // 1: the small-row tasks run on the key-tile tensor kernel
  int32_t tt_ctas;       // CTAs of the key-tile kernel (its task table's ranges)
};

// Host memory for plan tables.  Page-locked when a CUDA device is usable, so
// the upload in pps_attn_run is asynchronous and host planning of the next
// batch overlaps the GPU work of this one; ordinary memory otherwise.  A
// released buffer is handed out again only after the last upload recorded on
// it (host_buf_mark_use) has completed.
struct HostBuf {
  int32_t* data = nullptr;
  size_t ints = 0;
  int slot = -1;
};
HostBuf host_buf_acquire(size_t ints);
void host_buf_release(HostBuf& b);
int host_buf_mark_use(const HostBuf& b, void* stream);

}  // namespace pps

namespace pps {
// pps_attn_plan_tree, with the tensor-core tasks of requests [0, split_request)
// ordered first when split_request > 0 and the batch allows an output split
// (tensor-core tasks only, no shared-prefix groups, no partials); see
// pps_plan::num_mma_first.
pps_status plan_tree(const int32_t* q_indptr, const int32_t* kv_len, const int32_t* page_indptr,
                     const int32_t* page_indices, const int32_t* tree_parent,
                     int32_t num_requests, int32_t num_q_heads, int32_t num_kv_heads,
                     int32_t head_dim, int32_t page_size, int32_t num_pages, float sm_scale,
                     const pps_plan_options* opts, int32_t split_request, pps_plan** out_plan,
                     size_t* out_workspace_bytes);
}  // namespace pps

struct pps_plan {
  pps::Shape shape;
  int32_t num_requests = 0;
  int32_t num_tokens = 0;
  int32_t num_groups = 0;
  int64_t num_bw = 0, num_mma = 0, num_partials = 0, num_merge_tokens = 0, num_merge_pids = 0;
  // Output split (plans made with a split request only): the first
  // num_mma_first tensor-core tasks hold every row of the requests before
  // split_request and nothing else, so those rows (tokens [0, split_tokens))
  // are final once a launch over just those tasks has completed.  0: no split.
  int64_t num_mma_first = 0;
  int32_t split_tokens = 0;
  int64_t num_rows = 0, num_pages_listed = 0;
  int32_t num_tree_requests = 0;   // requests with a non-chain draft tree
  bool has_tree = false;           // table holds the per-token tree masks
  pps::TableLayout layout;
  pps::HostBuf image;           // host copy of the device table
  int64_t image_ints = 0;       // ints of the table in `image`
  size_t table_bytes = 0;       // bytes of the table, rounded to 256
  size_t partial_o_bytes = 0;
  size_t partial_lse_bytes = 0;
  size_t workspace_bytes = 0;
  mutable int64_t kv_bytes_unique = -1;   // computed on the first pps_plan_get_info
  int64_t kv_bytes_read = 0, kv_bytes_bw = 0;
  std::vector<int32_t> kv_len_copy, page_indptr_copy;   // inputs of that count
  int64_t tok_bytes = 0;
  double flops_mma_issued = 0;
  double flops_mma = 0, flops_total = 0;
  bool use_mma = false;
  ~pps_plan() { pps::host_buf_release(image); }
};

namespace pps {

// Kernel launchers (defined in the .cu files).  All return cudaSuccess (0) or
// the launch error.  `err` is the device error word of the current device.
// dst_slots: device int32 pairs {page, slot} per new token (8-byte aligned).
int launch_kv_append_slots(const pps_pool& pool, const void* k_new, const void* v_new,
                           const int32_t* dst_slots, int32_t num_new_tokens, void* stream);
int launch_kv_append(const pps_pool& pool, const void* k_new, const void* v_new,
                     const int32_t* q_indptr, const int32_t* cached_len,
                     const int32_t* page_indptr, const int32_t* page_indices,
                     int32_t num_requests, int32_t num_new_tokens, int32_t* err, void* stream);

int launch_copy_slots(const pps_pool& pool, const int32_t* src_pages, const int32_t* dst_pages,
                      const int32_t* num_slots, int32_t count, int32_t* err, void* stream);

int launch_gemm_bf16(const void* a, const void* w, void* c, int32_t M, int32_t N, int32_t K,
                     int32_t* err, void* stream);

// `app`: as launch_mma_attention; only the key-tile kernel (s.small_tt) takes it.
int launch_bw_attention(const Shape& s, const DeviceTables& t, int64_t num_tasks, const void* q,
                        const pps_pool& pool, void* out, int32_t* err, void* stream,
                        const AppendArgs* app = nullptr);

// `app` (may be null): the step's rows to append before any task reads the
// pool (one grid-wide wait; the kernel is then launched cooperatively).
int launch_mma_attention(const Shape& s, const DeviceTables& t, int64_t num_tasks, const void* q,
                         const pps_pool& pool, void* out, int32_t* err, void* stream,
                         const AppendArgs* app = nullptr);

// Small-row tasks (the bandwidth task list) on the key-tile tensor kernel.
int launch_tt_attention(const Shape& s, const DeviceTables& t, int64_t num_tasks, const void* q,
                        const pps_pool& pool, void* out, int32_t* err, void* stream,
                        const AppendArgs* app = nullptr);

int launch_merge(const Shape& s, const DeviceTables& t, int64_t num_merge_tokens, void* out,
                 void* stream);

bool mma_path_available();

#if defined(__CUDACC__)
}  // namespace pps
#include <cuda.h>
namespace pps {
// 4-D TMA view [num_pages][Hkv][P][D] of one pool array, box = 64 columns x P
// slots of one page and kv head, 128-byte swizzle (attn_mma.cu).
bool make_pool_map(CUtensorMap* map, const void* base, const pps_pool& pool);
#endif

#if defined(__CUDACC__)
// Launches `kern` on `stream` with programmatic stream serialization: it may
// start (and run its set-up) while the previous kernel of the stream is still
// running, and must call grid_dep_wait before it reads anything that kernel
// writes.  Without a kernel just before it in the stream it runs as usual.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem,
                             cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Launches `kern` cooperatively: every CTA is resident at once (or the launch
// fails), as a grid-wide wait inside the kernel requires.
template <typename... KArgs, typename... Args>
cudaError_t launch_cooperative(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem,
                               cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}
#endif

// SM count of the current device, or 0 when no device is usable.
int device_sm_count();

// Counts every kernel launch (pps_launch_count).
void count_launch();

}  // namespace pps
