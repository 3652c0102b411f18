// Tensor-core attention for tasks with few query rows: decode tokens, short
// verify drafts and shared-prefix groups of up to 32 rows (head_dim 128).
//
// The row-major tile (S = Q K^T with query rows on the MMA's M axis) needs 128
// query rows to fill the tensor core; a decode task has G of them.  Here the
// tile is transposed so the 128 KV positions of a tile sit on M and the task's
// (up to 32) query rows on N:
//     S^T[key, row]  = K[key, :] . Q[row, :]        (A = K tile, B = Q; both K-major)
//     O^T[d, row]   += V^T[d, key] . P^T[key, row]  (A = V tile MN-major, B = P^T MN-major)
// so every K/V byte streamed from HBM feeds one full-height MMA whatever the
// number of rows, and the CUDA cores only run the softmax (one exp per visible
// (key, row) pair).  The work is the XY-Serve review's matmul-softmax-matmul
// tile ("Core claim"; Fig. 10), with decode kept memory-bound as its Fig. 11
// describes, and the SGLang review's grouped shared-prefix rows ("Core claim")
// entering as up to 32 rows of one task.
//
// Warp roles (256 threads, one persistent CTA per SM running its own
// contiguous range of the task table, which the planner filled longest task
// first onto the least-loaded CTA):
//   warps 0-3  softmax: thread t owns TMEM lane t, i.e. key t of S^T and
//              element t of head_dim in O^T.  Per tile it reads its S^T lane
//              (32 rows), takes P = exp2(s * scale - m_ref[row]) against the
//              running reference max of every row (exact per-row maxima over
//              the 128 keys, and an O rescale in TMEM, only on a task's first
//              tile or when a score exceeds the reference by more than 2^8),
//              and writes its P^T row to shared memory as bf16 (64-byte
//              swizzle).  Epilogue: row sums reduced over the 128 threads, then
//              thread t writes element t of every row (or the fp32 partial).
//   warps 4,5  TMA producers of the K and of the V tiles of 128 positions (one
//              box per page and 64-column block) into 3-stage rings, 128-byte
//              swizzle.  K frees early (after QK) and V late (after PV), so each
//              ring refills on its own; page ids come from a 32-page window
//              prefetched one window ahead.
//   warp 6     MMA issuer: QK two tiles ahead of the softmax over the CTA's
//              whole tile stream (across tasks), PV of tile j once its P^T is
//              written.
//   warp 7     query rows of each task (cp.async, zero-filled past its rows)
//              into one of two 128-byte swizzled buffers, a task ahead.
// TMEM (128 columns): S^T_0 | S^T_1 | O^T_0 | O^T_1 (32 columns each); task i
// accumulates in O^T_(i & 1), so a task's output is written while the next
// task's first tile runs.  Every mbarrier
// wait is bounded; on timeout the kernel records PPS_DEV_ERR_WAIT_TIMEOUT,
// stops, drains what it issued and frees TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "pps_internal.h"
#include "sm100_ptx.cuh"
#include "append_dev.cuh"

namespace {

using namespace sm100;

constexpr int D = 128;
constexpr int kRows = pps::kTtRows;          // query rows per task = MMA N
constexpr int kTile = 128;                   // KV positions per tile = MMA M
constexpr int kStages = 3;
constexpr int kThreads = 256;
constexpr int kProducerK = 4;                // TMA of the K tiles
constexpr int kProducerV = 5;                // TMA of the V tiles
constexpr int kMmaWarp = 6;
constexpr int kQWarp = 7;                    // query rows of the next tasks
constexpr float kRescaleThreshold = 8.f;     // log2 units
constexpr uint64_t kLayoutSwizzle64 = 4;     // smem descriptor layout: 64-byte swizzle

struct TtParams {
  const pps::Task* tasks;
  const int32_t* cta_tasks;                  // CTA b runs tasks [cta_tasks[b], cta_tasks[b + 1])
  const int32_t* rows;
  const int32_t* pages;
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  float* o_part;
  float* lse_part;
  int32_t* err;
  const unsigned long long* tree_mask;       // per new token (draft trees), or nullptr
  int32_t num_q_heads;
  int32_t G;
  int32_t page_size;
  float qk_scale;                            // sm_scale * log2(e)
  // the step's rows to append first (num_tokens 0: none), into the pool
  pps::AppendArgs append;
  void* pool_k;
  void* pool_v;
  int32_t num_kv_heads;
  int32_t num_pages;
  int32_t* sync;
};

struct TtBars {
  uint64_t k_full[kStages], k_empty[kStages], v_full[kStages], v_empty[kStages];
  uint64_t q_full[2], q_empty[2], s_full[2], p_full[2], p_empty[2], o_done[2], drain;
};

// Shared memory (offsets from a 1024-byte aligned base).
struct TtLayout {
  static constexpr int kv_tile = 2 * 16384;             // 128 keys x 128 d, two 64-column blocks
  static constexpr int q_block = kRows * 128;           // 32 rows x 64 columns
  static constexpr int q_tile = 2 * q_block;
  static constexpr int p_tile = kTile * kRows * 2;      // 128 keys x 32 rows, bf16
  static constexpr int k_off = 0;
  static constexpr int v_off = k_off + kStages * kv_tile;
  static constexpr int q_off = v_off + kStages * kv_tile;
  static constexpr int p_off = q_off + 2 * q_tile;
  // per-row scratch: the tile maxima and (at a task's end) the row sums, one
  // use at a time: [kRows][4 warps] fp32
  static constexpr int red_off = p_off + 2 * p_tile;
  static constexpr int m_off = red_off + kRows * 4 * 4;         // reference max per row
  static constexpr int a_off = m_off + kRows * 4;               // rescale factor per row
  static constexpr int inv_off = a_off + kRows * 4;             // 1 / l per row of a finished task
  static constexpr int base_off = inv_off + kRows * 4;          // its output offset per row
  static constexpr int msk_off = base_off + kRows * 8;          // draft-tree masks per token
  static constexpr int bytes = msk_off + kRows * 8;
  static constexpr int smem_alloc = bytes + 1024;       // slack for the 1024-byte alignment
};
static_assert(TtLayout::smem_alloc + (int)sizeof(TtBars) + 64 <= 232448, "shared memory");

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The CTA's tasks (a contiguous range of the table, filled by the planner
// longest first onto the least-loaded CTA) in order, each record loaded one
// task ahead so that its global-memory latency overlaps the task before it.
struct TaskCursor {
  const pps::Task* tasks;
  int k, end;
  pps::Task nxt;
  __device__ __forceinline__ TaskCursor(const pps::Task* t, int lo, int hi)
      : tasks(t), k(lo), end(hi) {
    if (k < end) nxt = tasks[k];
  }
  __device__ __forceinline__ bool next(pps::Task& out) {
    if (k >= end) return false;
    out = nxt;
    if (++k < end) nxt = tasks[k];
    return true;
  }
};

__device__ __forceinline__ int n_tiles_of(const pps::Task& t) {
  return t.kv_end > t.kv_begin ? (t.kv_end - t.kv_begin + kTile - 1) / kTile : 0;
}

// OR of `pred` over the 128 softmax threads (named barrier 1).
__device__ __forceinline__ bool softmax_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n"
      " bar.red.or.pred po, 1, 128, pi;\n selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void softmax_sync() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Reduce-scatter of v[0..CUR) over lanes xor O, O/2, ..., 1 (max or sum):
// each halving step keeps one half and receives the partner's other half;
// once one value is left, the remaining lanes are folded in whole.  From
// CUR = NR, O = 16, lane l ends with the reduction of row rs_row<NR, 16>(l).
template <int CUR, int O, bool MAX>
__device__ __forceinline__ void reduce_scatter(float* v, int lane) {
  if constexpr (O >= 1) {
    if constexpr (CUR > 1) {
      constexpr int H = CUR / 2;
      const bool up = (lane & O) != 0;
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const float send = up ? v[i] : v[i + H];
        const float keep = up ? v[i + H] : v[i];
        const float got = __shfl_xor_sync(0xffffffffu, send, O);
        v[i] = MAX ? fmaxf(keep, got) : keep + got;
      }
      reduce_scatter<H, O / 2, MAX>(v, lane);
    } else {
      const float got = __shfl_xor_sync(0xffffffffu, v[0], O);
      v[0] = MAX ? fmaxf(v[0], got) : v[0] + got;
      reduce_scatter<1, O / 2, MAX>(v, lane);
    }
  }
}
template <int CUR, int O>
__device__ __forceinline__ int rs_row(int lane) {
  if constexpr (O >= 1 && CUR > 1) return ((lane & O) ? CUR / 2 : 0) + rs_row<CUR / 2, O / 2>(lane);
  else return 0;
}

// NR consecutive TMEM columns of the warp's 32 lanes.
template <int NR>
__device__ __forceinline__ void tm_ld(uint32_t a, uint32_t (&r)[NR]) {
  if constexpr (NR == 8) tmem_ld8(a, r);
  else if constexpr (NR == 16) tmem_ld16(a, r);
  else tmem_ld32(a, r);
}
template <int NR>
__device__ __forceinline__ void tm_st(uint32_t a, const uint32_t (&r)[NR]) {
  if constexpr (NR == 8) tmem_st8(a, r);
  else if constexpr (NR == 16) tmem_st16(a, r);
  else tmem_st32(a, r);
}

// What a softmax thread needs besides its task.
struct SmCtx {
  const TtParams* p;
  TtBars* bars;
  uint8_t* smem;
  float* red_max;                  // [kRows][4 warps]
  float* red_sum;
  int64_t* base_s;                 // [kRows] element offset of every output row of that task
  float* m_s;                      // [kRows] reference max of every row
  float* a_s;                      // [kRows] rescale factor of every row
  float* inv_s;                    // [kRows] 1 / l of every row of the last finished task
  unsigned long long* msk_s;       // [kRows] draft-tree lookback masks of the task's tokens
  volatile int* abort_flag;
  uint32_t tm, lane_off;
  int t, warp, lane;
};

__device__ __forceinline__ void sm_fail(const SmCtx& c) {
  atomicCAS(c.p->err, 0, PPS_DEV_ERR_WAIT_TIMEOUT);
  *c.abort_flag = 1;
}

// NR consecutive floats of shared memory (16-byte aligned) into registers.
template <int NR>
__device__ __forceinline__ void lds_rows(const float* src, float (&dst)[NR]) {
#pragma unroll
  for (int r = 0; r < NR; r += 4) {
    const float4 v = *reinterpret_cast<const float4*>(src + r);
    dst[r] = v.x;
    dst[r + 1] = v.y;
    dst[r + 2] = v.z;
    dst[r + 3] = v.w;
  }
}

// One task's tiles on the softmax warps, rows padded to NR (8, 16 or 32):
// every tile's S^T -> P^T; `after_first()` runs once the first tile's P^T is
// handed over (the previous task's output then overlaps this task's MMAs);
// then the task's row statistics: 1 / l per row (inv_s), lse of partial rows,
// output offsets (base_s).  gt counts tiles.  Returns false when a wait ran out
// (decided by all 128 threads together).  The per-tile path keeps its rows in
// registers; the rare paths (a task's first tile, a rescale, the statistics)
// work one row per lane and through shared memory, so they stay short in code
// as well as in time.
template <int NR, bool TREE, class AfterFirst>
__device__ __forceinline__ bool softmax_tiles(const SmCtx& c, const pps::Task& task, int n, int ti,
                                              int& gt, AfterFirst&& after_first) {
  const TtParams& p = *c.p;
  const int t = c.t, lane = c.lane, warp = c.warp, G = p.G;
  const int nrows = task.n_tok * G;
  const bool causal = task.causal != PPS_NO_CAUSAL;
  const uint32_t tm_o = c.tm + 2 * kRows + (ti & 1) * kRows;
  // The first tile takes the exact per-row maxima below, which set each row's
  // reference to its maximum (its largest P is then exactly 1); padding rows
  // see no key and keep a reference of 0, so their P stays 0.
  if (t < kRows) c.m_s[t] = 0.f;
  // token ids for the statistics step (loaded now, stored there)
  const int32_t my_tok = t < task.n_tok ? p.rows[task.row_off + t] : 0;
  // Draft trees: bit k of a token's mask = the key k positions before its own
  // one is visible (only new-token keys can be hidden; cached ones never are).
  if (TREE && t < task.n_tok) c.msk_s[t] = causal ? p.tree_mask[my_tok] : ~0ull;
  const int lg = __ffs(G) - 1;                           // G is a power of two
  float m_ref[NR], l_sum[NR];
#pragma unroll
  for (int r = 0; r < NR; ++r) {
    m_ref[r] = 0.f;
    l_sum[r] = 0.f;
  }
  if (n == 0 && !after_first()) return false;
  for (int j = 0; j < n; ++j, ++gt) {
    const int sb = gt & 1;
    const int t0 = task.kv_begin + j * kTile;
    bool got = mbar_wait_live(smem_u32(&c.bars->s_full[sb]), (gt >> 1) & 1, c.abort_flag);
    // the P^T buffer sb is free once the PV two tiles back has completed
    if (gt >= 2) got = got && mbar_wait(smem_u32(&c.bars->p_empty[sb]), ((gt - 2) >> 1) & 1);
    if (softmax_or(!got)) {
      if (t == 0) sm_fail(c);
      return false;
    }
    tc_fence_after();
    uint32_t s[NR];
    tm_ld<NR>(c.tm + c.lane_off + sb * kRows, s);
    tmem_wait_ld();
    const int pos = t0 + t;
    // no masking: every key valid and before every row's limit (before the first
    // new token for draft trees, whose own keys may be hidden)
    const int last_free = TREE ? task.causal - 1 : task.causal;
    const bool full = t0 + kTile <= task.kv_end && (!causal || t0 + kTile - 1 <= last_free);
    // row r (token r / G) sees key `pos` when r >= G * (pos - causal)
    const int first_vis = (full || !causal) ? 0 : G * (pos - task.causal);
    const bool key_ok = full || pos < task.kv_end;
    float x[NR];
    bool need = j == 0;
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      bool vis = r < nrows && key_ok && r >= first_vis;
      if (TREE && !full && causal && pos >= task.causal) {
        const int back = task.causal + (r >> lg) - pos;     // key `back` positions before row r's token
        if (back >= 0 && back < 64 && !((c.msk_s[r >> lg] >> back) & 1ull)) vis = false;
      }
      x[r] = vis ? __uint_as_float(s[r]) * p.qk_scale : -INFINITY;
      need |= x[r] > m_ref[r] + kRescaleThreshold;
    }
    if (softmax_or(need)) {
      // exact per-row maxima of this tile over its 128 keys; lane r of warp 0
      // then updates row r's reference and rescale factor
      {
        float v[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) v[r] = x[r];
        reduce_scatter<NR, 16, true>(v, lane);
        c.red_max[rs_row<NR, 16>(lane) * 4 + warp] = v[0];
      }
      softmax_sync();
      if (warp == 0 && lane < NR) {
        const float4 mm = *reinterpret_cast<const float4*>(c.red_max + lane * 4);
        const float mt = fmaxf(fmaxf(mm.x, mm.y), fmaxf(mm.z, mm.w));
        const float mo = c.m_s[lane];
        float mn = mo;
        if (j == 0) {
          if (mt != -INFINITY) mn = mt;      // first tile: the row's own maximum
        } else if (mt > mo + kRescaleThreshold) {
          mn = fmaxf(mt, mo);
        }
        c.a_s[lane] = j == 0 ? 1.f : ex2(mo - mn);   // nothing accumulated before the first tile
        c.m_s[lane] = mn;
      }
      softmax_sync();
      float alpha[NR];
      lds_rows<NR>(c.m_s, m_ref);
      lds_rows<NR>(c.a_s, alpha);
      bool resc = false;
#pragma unroll
      for (int r = 0; r < NR; ++r) {
        resc |= alpha[r] != 1.f;
        l_sum[r] *= alpha[r];
      }
      // Same values in every thread, so the branch is uniform.  O holds the
      // previous tiles' sum once the previous PV has completed.
      if (j > 0 && resc) {
        const bool g2 = mbar_wait(smem_u32(&c.bars->p_empty[(gt - 1) & 1]), ((gt - 1) >> 1) & 1) &&
                        !*c.abort_flag;
        if (softmax_or(!g2)) {
          if (t == 0) sm_fail(c);
          return false;
        }
        tc_fence_after();
        uint32_t o[NR];
        tm_ld<NR>(tm_o + c.lane_off, o);
        tmem_wait_ld();
#pragma unroll
        for (int r = 0; r < NR; ++r) o[r] = __float_as_uint(__uint_as_float(o[r]) * alpha[r]);
        tm_st<NR>(tm_o + c.lane_off, o);
        tmem_wait_st();
      }
    }
    // P^T row of key t: rows 0..NR-1 as bf16 (the first NR / 8 16-byte units
    // of its 64-byte row; units past them only feed O^T columns never read),
    // swizzled by the key's position in its 512-byte atom.
    uint32_t pk[NR / 2];
#pragma unroll
    for (int r = 0; r < NR; r += 2) {
      const float a = ex2(x[r] - m_ref[r]);          // references are always finite
      const float b = ex2(x[r + 1] - m_ref[r + 1]);
      l_sum[r] += a;
      l_sum[r + 1] += b;
      pk[r / 2] = pack_bf16(a, b);
    }
    uint8_t* pt = c.smem + TtLayout::p_off + sb * TtLayout::p_tile + t * 64;
#pragma unroll
    for (int u = 0; u < NR / 8; ++u)
      *reinterpret_cast<int4*>(pt + ((u ^ ((t >> 1) & 3)) << 4)) =
          make_int4((int)pk[4 * u], (int)pk[4 * u + 1], (int)pk[4 * u + 2], (int)pk[4 * u + 3]);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&c.bars->p_full[sb]));
    if (j == 0 && !after_first()) return false;
  }

  // ---- row statistics (no TMEM access: O may still be accumulating)
  {
    float v[NR];
#pragma unroll
    for (int r = 0; r < NR; ++r) v[r] = l_sum[r];
    reduce_scatter<NR, 16, false>(v, lane);
    c.red_sum[rs_row<NR, 16>(lane) * 4 + warp] = v[0];
  }
  softmax_sync();             // also: the previous task's output is done with inv_s, base_s
  // lane l of warp 0 holds token l: row r's token is lane r >> lg's
  const int row_tok = __shfl_sync(0xffffffffu, my_tok, (lane >> lg) & 31);
  if (warp == 0 && lane < NR) {
    // lane r: row r's 1 / l, its output offset (token or partial slot, head),
    // and its lse when the row is a partial
    const float4 ss = *reinterpret_cast<const float4*>(c.red_sum + lane * 4);
    const float lsum = (ss.x + ss.y) + (ss.z + ss.w);
    c.inv_s[lane] = lsum > 0.f ? 1.f / lsum : 0.f;
    const int i = lane >> lg, h = task.kv_head * G + (lane & (G - 1));
    const int64_t slot = task.out_pid < 0 ? (int64_t)row_tok : (int64_t)task.out_pid + i;
    c.base_s[lane] = (slot * p.num_q_heads + h) * D;
    if (task.out_pid >= 0 && lane < nrows)
      p.lse_part[slot * p.num_q_heads + h] = lsum > 0.f ? c.m_s[lane] + __log2f(lsum) : -INFINITY;
  }
  softmax_sync();
  return true;
}

// The output of a finished task (statistics in inv_s / base_s): once its last
// PV has completed, thread t writes element t of every row, O^T / l, as bf16
// (or the fp32 partial).  Rows in groups of 8 TMEM columns, so the code is the
// same for every row count.
__device__ __forceinline__ bool softmax_output(const SmCtx& c, const pps::Task& task, int ti) {
  const TtParams& p = *c.p;
  const int t = c.t;
  const int n = n_tiles_of(task), nrows = task.n_tok * p.G;
  bool got = true;
  if (n > 0) got = mbar_wait_live(smem_u32(&c.bars->o_done[ti & 1]), (ti >> 1) & 1, c.abort_flag);
  if (softmax_or(!got)) {
    if (t == 0) sm_fail(c);
    return false;
  }
  tc_fence_after();
  const uint32_t tm_o = c.tm + 2 * kRows + (ti & 1) * kRows + c.lane_off;
  const bool direct = task.out_pid < 0;
#pragma unroll 1
  for (int c0 = 0; c0 < nrows; c0 += 8) {
    uint32_t o[8];
    if (n > 0) {
      tmem_ld8(tm_o + c0, o);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int r = 0; r < 8; ++r) o[r] = 0u;
    }
#pragma unroll
    for (int r8 = 0; r8 < 8; ++r8) {
      const int r = c0 + r8;
      if (r < nrows) {
        const float val = __uint_as_float(o[r8]) * c.inv_s[r];
        if (direct)
          p.out[c.base_s[r] + t] = __float2bfloat16_rn(val);
        else
          p.o_part[c.base_s[r] + t] = val;
      }
    }
  }
  tc_fence_before();          // the O reads finish before this buffer's next first PV
  return true;
}

// TREE: the batch holds draft-tree verify rows; batches without one run the
// TREE = false instance, which has no mask code.
template <bool TREE>
__global__ void __launch_bounds__(kThreads, 1)
    tt_attention_kernel(const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const TtParams p) {
  using L = TtLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ TtBars bars;
  __shared__ uint32_t tmem_base;
  __shared__ volatile int abort_flag;
  __shared__ int task_range[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x;
  const int G = p.G;
  const uint32_t k_base = smem_u32(smem + L::k_off);
  const uint32_t v_base = smem_u32(smem + L::v_off);
  const uint32_t q_base = smem_u32(smem + L::q_off);
  const uint32_t p_base = smem_u32(smem + L::p_off);
  float* red_max = reinterpret_cast<float*>(smem + L::red_off);   // [kRows][4 warps]
  float* red_sum = red_max;                                       // (not live at once)
  int64_t* base_s = reinterpret_cast<int64_t*>(smem + L::base_off);  // [kRows]

  if (tid == 0) {
    const int lo = p.cta_tasks[b], hi = p.cta_tasks[b + 1];   // latency hidden by the set-up
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars.k_full[s]), 1);
      mbar_init(smem_u32(&bars.k_empty[s]), 1);
      mbar_init(smem_u32(&bars.v_full[s]), 1);
      mbar_init(smem_u32(&bars.v_empty[s]), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&bars.q_full[x]), 1);
      mbar_init(smem_u32(&bars.q_empty[x]), 1);
      mbar_init(smem_u32(&bars.s_full[x]), 1);
      mbar_init(smem_u32(&bars.p_full[x]), 4);
      mbar_init(smem_u32(&bars.p_empty[x]), 1);
    }
    for (int x = 0; x < 2; ++x) mbar_init(smem_u32(&bars.o_done[x]), 1);
    mbar_init(smem_u32(&bars.drain), 1);
    abort_flag = 0;
    task_range[0] = lo;
    task_range[1] = hi;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&tmem_base), 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = tmem_base;
  const uint32_t tm_o = tm + 2 * kRows;
  // Set-up done: let the next kernel of the stream be scheduled, then wait
  // for the one before (the append writes the pool rows this kernel reads).
  grid_dep_launch();
  grid_dep_wait();
  // The step's new K/V rows, when this launch carries the append: every CTA
  // copies its share, then all wait for one another before any task reads
  // the pool.
  if (p.append.num_tokens > 0) {
    pps_dev::append_rows<D>(p.append, reinterpret_cast<int4*>(p.pool_k),
                            reinterpret_cast<int4*>(p.pool_v), p.num_kv_heads, p.page_size,
                            p.num_pages, p.err, warp, lane, kThreads / 32);
    pps_dev::grid_wait(p.sync, p.err);
  }

  auto fail = [&]() {
    atomicCAS(p.err, 0, PPS_DEV_ERR_WAIT_TIMEOUT);
    abort_flag = 1;
  };
  auto warp_wait = [&](uint64_t* bar, uint32_t parity, bool needed = true) -> bool {
    if (__all_sync(0xffffffffu, !needed || mbar_try_wait(smem_u32(bar), parity))) return true;
    const bool ok = (!needed || mbar_wait(smem_u32(bar), parity)) && !abort_flag;
    return __all_sync(0xffffffffu, ok) != 0;
  };

  if (warp < 4) {
    // ------------------------------------------------------------- softmax warps
    const int t = tid;                                   // TMEM lane: key t / element t
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    SmCtx ctx{&p,      &bars,         smem,     red_max, red_sum, base_s,
              reinterpret_cast<float*>(smem + L::m_off), reinterpret_cast<float*>(smem + L::a_off),
              reinterpret_cast<float*>(smem + L::inv_off),
              reinterpret_cast<unsigned long long*>(smem + L::msk_off), &abort_flag, tm, lane_off,
              t, warp, lane};
    TaskCursor cur(p.tasks, task_range[0], task_range[1]);
    pps::Task task, prev;
    int prev_ti = -1;                                    // finished task whose output is pending
    int gt = 0;                                          // tiles seen
    bool ok = true;
    for (int ti = 0; cur.next(task); ++ti) {
      const int n = n_tiles_of(task);
      const int nrows = task.n_tok * G;
      auto flush = [&]() -> bool {
        if (prev_ti < 0) return true;
        const int pt = prev_ti;
        prev_ti = -1;
        return softmax_output(ctx, prev, pt);
      };
      // rows padded to 8, 16 or 32 (uniform over the CTA: one task at a time)
      if (nrows <= 8) ok = softmax_tiles<8, TREE>(ctx, task, n, ti, gt, flush);
      else if (nrows <= 16) ok = softmax_tiles<16, TREE>(ctx, task, n, ti, gt, flush);
      else ok = softmax_tiles<32, TREE>(ctx, task, n, ti, gt, flush);
      if (!ok) break;
      prev = task;
      prev_ti = ti;
    }
    if (ok && prev_ti >= 0) softmax_output(ctx, prev, prev_ti);
  } else if (warp == kQWarp) {
    // ------------------------------------------------------------ query rows
    // Task ti's rows go to buffer ti & 1 once the QKs of task ti - 2 (the
    // buffer's previous user) have completed: 32 rows x 256 bytes, 16 bytes
    // per copy, 128-byte swizzled K-major, zeros past the task's rows.
    bool ok = true;
    TaskCursor cur(p.tasks, task_range[0], task_range[1]);
    pps::Task task;
    for (int ti = 0; ok && cur.next(task); ++ti) {
      const int qb = ti & 1;
      const bool freed = ti < 2 || mbar_wait_idle(smem_u32(&bars.q_empty[qb]), ((ti >> 1) - 1) & 1);
      if (!__all_sync(0xffffffffu, freed && !abort_flag)) { fail(); ok = false; break; }
      const int nrows = task.n_tok * G;
      const int my_tok = lane < task.n_tok ? p.rows[task.row_off + lane] : 0;
      const uint32_t qt = q_base + qb * L::q_tile;
#pragma unroll 4
      for (int c = lane; c < kRows * 16; c += 32) {
        const int r = c >> 4, u = c & 15;
        const int i = r / G, h = task.kv_head * G + (r - i * G);
        const int tok = __shfl_sync(0xffffffffu, my_tok, i & 31);
        const bool real = r < nrows;
        cp_async16(qt + (u >> 3) * L::q_block + sw128(r, u & 7),
                   real ? (const void*)(p.q + ((size_t)tok * p.num_q_heads + h) * D + u * 8)
                        : (const void*)p.q,
                   real ? 16u : 0u);
      }
      cp_async_wait_all();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars.q_full[qb]));
    }
  } else if (warp == kProducerK || warp == kProducerV) {
    // ------------------------------------------------------------ TMA producers
    const bool is_k = warp == kProducerK;
    const CUtensorMap* map = is_k ? &tmk : &tmv;
    uint64_t* full = is_k ? bars.k_full : bars.v_full;
    uint64_t* empty = is_k ? bars.k_empty : bars.v_empty;
    const uint32_t ring = is_k ? k_base : v_base;
    if (lane == 0) prefetch_tmap(map);
    const int P = p.page_size;
    const int ppt = kTile / P;                      // pages per tile (divides 32)
    const uint32_t box_bytes = (uint32_t)P * 128u;
    int it = 0;
    bool ok = true;
    TaskCursor cur(p.tasks, task_range[0], task_range[1]);
    pps::Task task;
    for (int ti = 0; ok && cur.next(task); ++ti) {
      const int n = n_tiles_of(task);
      // the task's pages from kv_begin (a multiple of P), 32 at a time: lane l
      // holds page wbase + l of `win`, and page wbase + 32 + l of `nxt`
      const int npages = n > 0 ? (task.kv_end - task.kv_begin + P - 1) / P : 0;
      const int32_t* pl = p.pages + task.page_off + task.kv_begin / P;
      int wbase = 0;
      int win = lane < npages ? pl[lane] : 0;
      int nxt = lane + 32 < npages ? pl[lane + 32] : 0;
      for (int j = 0; j < n; ++j, ++it) {
        const int st = it % kStages, use = it / kStages;
        const int rel0 = j * ppt;                   // the tile's first page in the task
        if (rel0 >= wbase + 32) {
          wbase += 32;
          win = nxt;
          nxt = lane + wbase + 32 < npages ? pl[lane + wbase + 32] : 0;
        }
        const int valid = min(kTile, task.kv_end - (task.kv_begin + j * kTile));
        const int npg = (valid + P - 1) / P;
        const int pg = lane >> 1, kb = lane & 1;
        const int page = __shfl_sync(0xffffffffu, win, (rel0 - wbase + pg) & 31);
        const bool mine = lane < npg * 2;
        const uint32_t fb = smem_u32(&full[st]);
        if (!warp_wait(&empty[st], (use - 1) & 1, use > 0)) { fail(); ok = false; break; }
        if (lane == 0) mbar_expect_tx(fb, (uint32_t)(npg * 2) * box_bytes);
        __syncwarp();
        if (mine)
          tma_load_4d(ring + st * L::kv_tile + kb * 16384 + pg * P * 128, map, kb * 64, 0,
                      task.kv_head, page, fb);
      }
    }
    // every load this warp started lands before the CTA may exit
    if (lane == 0) {
      const uint64_t lim = ok ? 2000000000ull : 10000000ull;
      for (int j = (it > kStages ? it - kStages : 0); j < it; ++j)
        mbar_wait(smem_u32(&full[j % kStages]), (j / kStages) & 1, lim);
    }
  } else {
    // ------------------------------------------------------------- MMA issuer
    constexpr uint32_t id_qk = idesc_bf16(kTile, kRows, 0, 0);
    constexpr uint32_t id_pv = idesc_bf16(D, kRows, 1, 1);
    int gt = 0;
    bool ok = true;
    // S^T_(g & 1) = K_g Q^T; frees K_g.
    auto qk = [&](int g, int qb) -> bool {
      const int st = g % kStages;
      if (!warp_wait(&bars.k_full[st], (g / kStages) & 1)) return false;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t kd = smem_desc(k_base + st * L::kv_tile, 16, 1024);
        const uint64_t qd = smem_desc(q_base + qb * L::q_tile, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t ka = (ks / 4) * 16384 + (ks % 4) * 32;
          const uint32_t qa = (ks / 4) * L::q_block + (ks % 4) * 32;
          umma_ss(tm + (g & 1) * kRows, kd + (ka >> 4), qd + (qa >> 4), id_qk, ks > 0);
        }
        umma_commit(smem_u32(&bars.s_full[g & 1]));
        umma_commit(smem_u32(&bars.k_empty[st]));
      }
      __syncwarp();
      return true;
    };
    // A tile with `valid` < 128 keys runs only the PV steps (16 keys each)
    // that hold a valid key; the rest would multiply P = 0 by V rows that were
    // not loaded.  Inside the last step, rows from `valid` to the next multiple
    // of 16 are pool slots past the task's last position (the same page) and
    // may hold anything, NaN included: 0 * NaN would poison O, so they are
    // cleared (at most 15 rows of both 64-column blocks; whole 128-byte rows,
    // so the swizzle does not matter).
    auto clear_v_rows = [&](int st, int valid) {
      uint8_t* vt = smem + L::v_off + st * L::kv_tile;
      const int nch = (((valid + 15) & ~15) - valid) * 8;   // 16-byte chunks per block
#pragma unroll
      for (int kb = 0; kb < 2; ++kb)
        for (int i = lane; i < nch; i += 32)
          *reinterpret_cast<int4*>(vt + kb * 16384 + (valid + (i >> 3)) * 128 + (i & 7) * 16) =
              make_int4(0, 0, 0, 0);
      fence_proxy_async_smem();
      __syncwarp();
    };
    // QK runs two tiles ahead of PV over the CTA's whole tile stream, across
    // task boundaries: the next task's first S is ready when the softmax
    // finishes the current task.  `qc` walks the tasks for QK (waiting for
    // each task's query rows), `pc` for PV.
    TaskCursor qc(p.tasks, task_range[0], task_range[1]);
    pps::Task qtask{};
    int q_ti = -1, q_n = 0, q_j = 0;                // task, its tiles, next tile to QK
    int gq = 0;                                     // next global tile to QK
    // QK of global tile gq; false when the stream has ended or a wait ran out
    // (ok says which).
    auto qk_next = [&]() -> bool {
      while (q_j >= q_n) {
        if (!qc.next(qtask)) return false;
        ++q_ti;
        q_n = n_tiles_of(qtask);
        q_j = 0;
        if (!warp_wait(&bars.q_full[q_ti & 1], (q_ti >> 1) & 1)) {
          fail();
          ok = false;
          return false;
        }
        if (q_n == 0) {                             // no QK reads the buffer
          if (elect_one()) umma_commit(smem_u32(&bars.q_empty[q_ti & 1]));
          __syncwarp();
        }
      }
      if (!qk(gq, q_ti & 1)) {
        fail();
        ok = false;
        return false;
      }
      if (q_j == q_n - 1) {                         // the task's last QK: its buffer frees
        if (elect_one()) umma_commit(smem_u32(&bars.q_empty[q_ti & 1]));
        __syncwarp();
      }
      ++q_j;
      ++gq;
      return true;
    };
    while (gq < 2 && qk_next()) {
    }
    TaskCursor pc(p.tasks, task_range[0], task_range[1]);
    pps::Task task;
    for (int ti = 0; ok && pc.next(task); ++ti) {
      const int n = n_tiles_of(task);
      const int ob = ti & 1;
      if (n == 0) {                                 // nothing accumulated: O is ready now
        if (elect_one()) umma_commit(smem_u32(&bars.o_done[ob]));
        __syncwarp();
        continue;
      }
      for (int j = 0; j < n; ++j) {
        const int g = gt + j, sb = g & 1, st = g % kStages;
        if (!warp_wait(&bars.p_full[sb], (g >> 1) & 1)) { fail(); ok = false; break; }
        if (!warp_wait(&bars.v_full[st], (g / kStages) & 1)) { fail(); ok = false; break; }
        const int valid = min(kTile, task.kv_end - (task.kv_begin + j * kTile));
        const int nks = (valid + 15) >> 4;              // PV steps holding a valid key
        if (valid & 15) clear_v_rows(st, valid);
        tc_fence_after();
        if (elect_one()) {
          const uint64_t vd = smem_desc(v_base + st * L::kv_tile, 16384, 1024);
          const uint64_t pd = smem_desc(p_base + sb * L::p_tile, 1024, 512, kLayoutSwizzle64);
          if (nks == kTile / 16) {                  // whole tile: back-to-back issue
#pragma unroll
            for (int ks = 0; ks < kTile / 16; ++ks)
              umma_ss(tm_o + ob * kRows, vd + (uint64_t)(ks * 128), pd + (uint64_t)(ks * 64),
                      id_pv, (j > 0 || ks > 0) ? 1u : 0u);
          } else {
#pragma unroll 1
            for (int ks = 0; ks < nks; ++ks)
              umma_ss(tm_o + ob * kRows, vd + (uint64_t)(ks * 128), pd + (uint64_t)(ks * 64),
                      id_pv, (j > 0 || ks > 0) ? 1u : 0u);
          }
          umma_commit(smem_u32(&bars.v_empty[st]));
          umma_commit(smem_u32(&bars.p_empty[sb]));
          if (j == n - 1) umma_commit(smem_u32(&bars.o_done[ob]));
        }
        __syncwarp();
        // S buffer (g & 1) is free again: QK of tile g + 2, whichever task
        while (ok && gq <= g + 2 && qk_next()) {
        }
        if (!ok) break;
      }
      gt += n;
    }
    // Every MMA this warp issued has completed before TMEM is freed.
    if (elect_one()) {
      umma_commit(smem_u32(&bars.drain));
      if (!mbar_wait(smem_u32(&bars.drain), 0)) fail();
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tm, 128);
  }
}

}  // namespace

namespace pps {

namespace {
template <bool TREE>
int launch_tt(const Shape& s, const DeviceTables& t, const void* q, const pps_pool& pool,
              void* out, int32_t* err, void* stream, const AppendArgs* app) {
  CUtensorMap mk, mv;
  if (!make_pool_map(&mk, pool.k, pool) || !make_pool_map(&mv, pool.v, pool))
    return (int)cudaErrorInvalidValue;
  // once per device and instance: the shared-memory opt-in
  static std::atomic<int> ready[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  if (dev < 0 || dev >= 64 || !ready[dev].load(std::memory_order_relaxed)) {
    if ((e = cudaFuncSetAttribute(tt_attention_kernel<TREE>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  TtLayout::smem_alloc)) != cudaSuccess)
      return (int)e;
    if (dev >= 0 && dev < 64) ready[dev].store(1, std::memory_order_relaxed);
  }
  // one CTA per range of the plan's table (the planner sized them for the SMs)
  const int64_t grid = s.tt_ctas;
  if (grid <= 0 || !t.tt_cta) return (int)cudaErrorInvalidValue;
  TtParams prm{t.bw_tasks, t.tt_cta, t.rows, t.pages, (const __nv_bfloat16*)q,
               (__nv_bfloat16*)out, t.o_part, t.lse_part, err, t.tree_mask, s.num_q_heads,
               s.group, s.page_size, s.sm_scale * 1.4426950408889634f,
               app ? *app : AppendArgs{}, pool.k, pool.v, pool.num_kv_heads, pool.num_pages,
               t.sync};
  // with the append every CTA must be resident at once (it waits for all)
  e = app ? launch_cooperative(tt_attention_kernel<TREE>, (unsigned)grid, kThreads,
                               TtLayout::smem_alloc, (cudaStream_t)stream, mk, mv, prm)
          : launch_dependent(tt_attention_kernel<TREE>, (unsigned)grid, kThreads,
                             TtLayout::smem_alloc, (cudaStream_t)stream, mk, mv, prm);
  count_launch();
  return (int)e;
}
}  // namespace

int launch_tt_attention(const Shape& s, const DeviceTables& t, int64_t num_tasks, const void* q,
                        const pps_pool& pool, void* out, int32_t* err, void* stream,
                        const AppendArgs* app) {
  if (num_tasks == 0) return cudaSuccess;
  if (s.head_dim != D) return (int)cudaErrorInvalidValue;
  return t.tree_mask ? launch_tt<true>(s, t, q, pool, out, err, stream, app)
                     : launch_tt<false>(s, t, q, pool, out, err, stream, app);
}

}  // namespace pps
