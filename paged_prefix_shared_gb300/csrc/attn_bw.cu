// Bandwidth-path attention: split-KV tasks with few query rows (decode rows,
// small shared-prefix groups), fp32 math on CUDA cores.
//
// Decode attention is a matrix-vector product and memory bound (XY-Serve
// review, Fig. 11 "mask-aware computation" caption); long KV is split into
// chunks whose partial softmax results are merged afterwards (online softmax
// equals softmax, "Assumptions & free parameters").  Each CTA runs one task:
// all query rows (tokens x the G query heads of one kv head) against one KV
// chunk of one page list, so every K/V byte of the chunk is read once for all
// G heads, and once for every member of a shared-prefix group.
//
// Per block of kKB positions: (1) scores, lanes split head_dim and reduce with
// warp shuffles; (2) per-row block max / rescale / exp2 in shared memory;
// (3) P.V accumulated in registers.  A final cross-warp reduction writes the
// bf16 output row or an fp32 partial (o normalised, lse in log2 units).
#include <cuda_bf16.h>
#include <algorithm>
#include <cuda_runtime.h>

#include "pps_internal.h"
#include "sm100_ptx.cuh"

namespace {

constexpr int kThreads = 128;
constexpr int kKB = 256;                      // KV positions per block
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void bf16x8_to_f32(const int4& v, float* f) {
  const uint32_t w[4] = {(uint32_t)v.x, (uint32_t)v.y, (uint32_t)v.z, (uint32_t)v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <int D, int R>
__global__ void __launch_bounds__(kThreads) bw_attention_kernel(
    const pps::Task* __restrict__ tasks, const int32_t* __restrict__ rows,
    const int32_t* __restrict__ pages, const __nv_bfloat16* __restrict__ q,
    const __nv_bfloat16* __restrict__ pool_k, const __nv_bfloat16* __restrict__ pool_v,
    __nv_bfloat16* __restrict__ out, float* __restrict__ o_part, float* __restrict__ lse_part,
    const unsigned long long* __restrict__ tree_mask, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t G, int32_t page_size, float qk_scale) {
  constexpr int LPT = D / 8;                  // lanes per KV row (8 bf16 = 16 B each)
  constexpr int TPI = kThreads / LPT;         // KV rows per CTA iteration
  extern __shared__ float smem[];
  float* m_run = smem;                        // [R] running max (log2 units)
  float* l_run = smem + R;                    // [R] running sum
  float* alpha = smem + 2 * R;                // [R] rescale factor of the current block
  float* s = smem + 4 * R;                    // [R][kKB] scores / probabilities
  float* red = s;                             // reused at the end: [4 warps][R][D]

  const pps::Task task = tasks[blockIdx.x];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tok = tid / LPT;                  // which KV row of the iteration
  const int dl = (tid % LPT) * 8;             // first head_dim column of this lane
  const int nrows = task.n_tok * G;
  const int h0 = task.kv_head * G;

  // Query rows (row r = token r / G, query head h0 + r % G), pre-scaled to log2 units.
  float qr[R][8];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (r < nrows) {
      const int t = rows[task.row_off + r / G];
      const int4 v = *reinterpret_cast<const int4*>(q + ((size_t)t * num_q_heads + h0 + r % G) * D + dl);
      bf16x8_to_f32(v, qr[r]);
#pragma unroll
      for (int e = 0; e < 8; ++e) qr[r][e] *= qk_scale;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) qr[r][e] = 0.f;
    }
  }
  if (tid < R) { m_run[tid] = -INFINITY; l_run[tid] = 0.f; }
  // Draft-tree lookback masks of the task's tokens (all ones: plain causal).
  __shared__ unsigned long long tmk[R];
  if (tid < R)
    tmk[tid] = (tree_mask && tid < task.n_tok && task.causal != PPS_NO_CAUSAL)
                   ? tree_mask[rows[task.row_off + tid]] : ~0ull;
  __syncthreads();
  float acc[R][8];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[r][e] = 0.f;

  const size_t head_stride = (size_t)page_size * D;
  auto row_ptr = [&](const __nv_bfloat16* base, int p) {
    const int page = pages[task.page_off + p / page_size];
    return base + ((size_t)page * num_kv_heads + task.kv_head) * head_stride +
           (size_t)(p % page_size) * D + dl;
  };

  for (int b0 = task.kv_begin; b0 < task.kv_end; b0 += kKB) {
    const int nb = min(kKB, task.kv_end - b0);
    // (1) scores
    for (int i0 = 0; i0 < nb; i0 += TPI) {     // trip count uniform across the CTA
      const int i = i0 + tok;
      const bool in = i < nb;
      const int p = b0 + (in ? i : 0);
      float k[8];
      bf16x8_to_f32(__ldg(reinterpret_cast<const int4*>(row_ptr(pool_k, p))), k);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float d = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) d = fmaf(qr[r][e], k[e], d);
#pragma unroll
        for (int off = LPT / 2; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
        if (in && dl == 0 && r < nrows) {
          const int back = task.causal + r / G - p;        // keys before the row's own one
          const bool vis = back >= 0 && (back >= 64 || ((tmk[r / G] >> back) & 1ull));
          s[r * kKB + i] = vis ? d : -INFINITY;
        }
      }
    }
    __syncthreads();
    // (2) block max, rescale factor, probabilities
    for (int r = warp; r < nrows; r += 4) {
      float mb = -INFINITY;
      for (int i = lane; i < nb; i += 32) mb = fmaxf(mb, s[r * kKB + i]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
      const float mo = m_run[r];
      const float mn = fmaxf(mo, mb);
      const float ms = (mn == -INFINITY) ? 0.f : mn;    // row saw nothing yet: keep zeros
      float lb = 0.f;
      for (int i = lane; i < nb; i += 32) {
        const float pr = exp2f(s[r * kKB + i] - ms);
        s[r * kKB + i] = pr;
        lb += pr;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) lb += __shfl_xor_sync(0xffffffffu, lb, off);
      __syncwarp();
      if (lane == 0) {
        const float a = (mo == -INFINITY) ? 0.f : exp2f(mo - ms);
        alpha[r] = a;
        m_run[r] = mn;
        l_run[r] = l_run[r] * a + lb;
      }
    }
    __syncthreads();
    // (3) P.V
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float a = (r < nrows) ? alpha[r] : 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[r][e] *= a;
    }
    for (int i = tok; i < nb; i += TPI) {
      float v[8];
      bf16x8_to_f32(__ldg(reinterpret_cast<const int4*>(row_ptr(pool_v, b0 + i))), v);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (r < nrows) {
          const float pr = s[r * kKB + i];
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[r][e] = fmaf(pr, v[e], acc[r][e]);
        }
      }
    }
    __syncthreads();
  }

  // Reduce the per-KV-row-slot accumulators: within the warp, then across warps.
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int e = 0; e < 8; ++e)
#pragma unroll
      for (int off = LPT; off < 32; off <<= 1)
        acc[r][e] += __shfl_xor_sync(0xffffffffu, acc[r][e], off);
  if (lane < LPT) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int e = 0; e < 8; ++e) red[(warp * R + r) * D + dl + e] = acc[r][e];
  }
  __syncthreads();
  for (int idx = tid; idx < nrows * D; idx += kThreads) {
    const int r = idx / D, c = idx % D;
    const float o = red[(0 * R + r) * D + c] + red[(1 * R + r) * D + c] +
                    red[(2 * R + r) * D + c] + red[(3 * R + r) * D + c];
    const float l = l_run[r];
    const float val = l > 0.f ? o / l : 0.f;
    const int i = r / G, h = h0 + r % G;
    if (task.out_pid < 0) {
      const int t = rows[task.row_off + i];
      out[((size_t)t * num_q_heads + h) * D + c] = __float2bfloat16_rn(val);
    } else {
      const size_t prow = (size_t)(task.out_pid + i) * num_q_heads + h;
      o_part[prow * D + c] = val;
      if (c == 0) lse_part[prow] = l > 0.f ? m_run[r] + log2f(l) : -INFINITY;
    }
  }
}

// ---------------------------------------------------------------------------
// Pipelined, persistent kernel (tasks of up to 8 query rows).
//
// One CTA per SM (8 warps: 7 consumers + 1 producer) loops over its share of
// the work-sorted task list.  The producer streams each task's query rows and
// its K and V rows 16 positions at a time (2 x 16 x d x 2 bytes per stage; a
// page of P >= 16 slots is P/16 sub-blocks) with cp.async.bulk into a
// 16-stage ring, running ahead across task boundaries.  Consumer warps take a
// task's sub-blocks round robin.  In a consumer warp, LPT lanes share one KV
// row (EL head_dim elements each, 16-byte chunks at stride LPT so shared
// memory reads are conflict free) and TPW rows are processed per step.  The R
// partial dot products of a lane are reduce-scattered across its LPT lanes
// (log2(LPT) shuffles in all, each lane ends with the full score of one
// row), the online softmax keeps a per-warp reference max (rescaled only when
// it rises by more than 2^8), and P.V accumulates in registers with packed
// fp32x2 FMAs.  The warps' states are merged through shared memory per task.

constexpr int kBw2Sub = 16;                   // KV positions per stage
constexpr int kBw2Consumers = 7;
// Every consumer warp owns kStagesPerWarp ring stages: sub-block g of the
// CTA's stream goes to warp g % kBw2Consumers, stage (g / kBw2Consumers) %
// kStagesPerWarp of that warp.  With one consumer per stage, waiting in order,
// a stage's full barrier is never waited on more than one phase ahead (its
// parity bit alone then identifies the phase).
constexpr int kStagesPerWarp = 3;
constexpr int kBw2Stages = kBw2Consumers * kStagesPerWarp;
constexpr int kBw2Threads = (kBw2Consumers + 1) * 32;
constexpr int kIssueLanes = 8;                // producer lanes issuing copies at once

template <int D, int R>
struct Bw2 {
  static constexpr int EL = (R >= 8) ? 8 : 16;            // head_dim elements per lane
  static constexpr int LPT = D / EL;                      // lanes per KV row
  static constexpr int TPW = 32 / LPT;                    // KV rows per warp step
  static constexpr int ITERS = kBw2Sub / TPW;
  static constexpr int CH = EL / 8;                       // 16-byte chunks per lane
  static constexpr int STAGE = 2 * kBw2Sub * D * 2;       // K then V
  static_assert(R <= LPT, "one row per lane after the reduce-scatter");
};

// Reduce-scatter of V[0..CUR) over lanes xor O, O/2, ..., 1: each halving step
// sends half of the values to the partner lane and keeps the other half.
template <int CUR, int O>
__device__ __forceinline__ void reduce_scatter(float* v, int lane) {
  if constexpr (O >= 1) {
    if constexpr (CUR > 1) {
      constexpr int H = CUR / 2;
      const bool up = (lane & O) != 0;
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const float send = up ? v[i] : v[i + H];
        const float keep = up ? v[i + H] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
      }
      reduce_scatter<H, O / 2>(v, lane);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
      reduce_scatter<1, O / 2>(v, lane);
    }
  }
}
// Row whose full score lane `lane` holds after reduce_scatter<R, LPT/2>.
template <int CUR, int O>
__device__ __forceinline__ int rs_row(int lane) {
  if constexpr (O >= 1 && CUR > 1) return ((lane & O) ? CUR / 2 : 0) + rs_row<CUR / 2, O / 2>(lane);
  else return 0;
}
// Lane (within its LPT group) that holds row r.
template <int R, int LPT>
__device__ __forceinline__ int rs_lane(int r) {
  int l = 0;
#pragma unroll
  for (int k = 1; (R >> k) >= 1; ++k)
    if (r & (R >> k)) l += LPT >> k;
  return l;
}

__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Persistent CTAs: CTA b takes tasks b, 2C-1-b, 2C+b, 4C-1-b, ... of the
// work-sorted list (symmetric round robin over C CTAs, the assignment the
// XY-Serve review's "What carries the argument" describes for sorted tiles).
__device__ __forceinline__ int snake_task(int ti, int b, int C) {
  return ti * C + ((ti & 1) ? (C - 1 - b) : b);
}

template <int D, int R>
struct Bw3Smem {
  using C = Bw2<D, R>;
  static constexpr int ring = 0;
  static constexpr int qbuf = kBw2Stages * C::STAGE;             // 2 x [R][D] bf16
  static constexpr int qbuf_bytes = R * D * 2;
  static constexpr int comb = qbuf + 2 * ((qbuf_bytes + 127) / 128 * 128);
  static constexpr int comb_bytes = kBw2Consumers * R * (D + 2) * 4;
  static constexpr int total = comb + comb_bytes;
};

// Pointers a consumer warp needs besides its task (shared memory of the CTA).
struct BwShared {
  const uint8_t* ring;
  uint64_t* full;
  uint64_t* empty;
  volatile int* abort_flag;
  int32_t* err;
  float* cm;
  float* cl;
  float* co;
};

// One consumer warp's share of one task: its sub-blocks (stream positions
// g = gk + k with g % kBw2Consumers == warp), an online softmax over the
// task's R rows, then its (max, sum, o) written to the combine buffer whose row
// stride is RS >= R.  Returns false when a wait ran out.
template <int D, int R, int RS, bool TREE>
__device__ __forceinline__ bool bw_consume(const pps::Task& task, int nrows, int G, int n_sub,
                                           int gk, const uint8_t* qs,
                                           const unsigned long long* tmk, float qk_scale,
                                           bool live, const BwShared& sh, uint64_t* qempty) {
  using C = Bw2<D, R>;
  constexpr int EL = C::EL, LPT = C::LPT, TPW = C::TPW, ITERS = C::ITERS, CH = C::CH;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = lane / LPT, sub = lane % LPT;
  const int my_row = rs_row<R, LPT / 2>(lane);
  float qr[R][EL];
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      float f[8];
      const int4 v = (live && r < nrows)
                         ? *reinterpret_cast<const int4*>(qs + r * D * 2 + (sub + j * LPT) * 16)
                         : make_int4(0, 0, 0, 0);
      bf16x8_to_f32(v, f);
#pragma unroll
      for (int x = 0; x < 8; ++x) qr[r][j * 8 + x] = f[x] * qk_scale;
    }
  }
  __syncwarp();
  if (lane == 0) sm100::mbar_arrive(sm100::smem_u32(qempty));

  float m_run = -INFINITY, l_run = 0.f;
  float acc[R][EL];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int e = 0; e < EL; ++e) acc[r][e] = 0.f;
  const int my_lim = task.causal + my_row / G;
  // Draft-tree tasks (TREE) mask non-ancestor keys among the 64 before each
  // row's own one; a sub-block takes the fast (unmasked) path only if it ends
  // before every row's window.
  unsigned long long my_mask = ~0ull;
  if constexpr (TREE) my_mask = (live && my_row < nrows) ? tmk[my_row / G] : ~0ull;
  const int lim0 = task.causal - (TREE ? 64 : 0);
  const int first = (warp - gk % kBw2Consumers + kBw2Consumers) % kBw2Consumers;
  for (int k = first; live && k < n_sub; k += kBw2Consumers) {
    const int g = gk + k;                                  // g % kBw2Consumers == warp
    const int wi = g / kBw2Consumers;
    const int s = warp * kStagesPerWarp + wi % kStagesPerWarp;
    const bool got =
        sm100::mbar_wait_live(sm100::smem_u32(&sh.full[s]), (wi / kStagesPerWarp) & 1, sh.abort_flag);
    if (!__all_sync(0xffffffffu, got)) {
      if (lane == 0) {
        atomicCAS(sh.err, 0, PPS_DEV_ERR_WAIT_TIMEOUT);
        *sh.abort_flag = 1;
      }
      live = false;
      break;
    }
    const int pos0 = task.kv_begin + k * kBw2Sub;
    const bool fast = (pos0 + kBw2Sub <= task.kv_end) && (pos0 + kBw2Sub - 1 <= lim0);
    const uint8_t* kb = sh.ring + s * (2 * kBw2Sub * D * 2);
    const uint8_t* vb = kb + kBw2Sub * D * 2;
    float sc[ITERS];
#pragma unroll
    for (int it = 0; it < ITERS; ++it) {
      const int tt = it * TPW + grp;
      float kf[EL];
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        const int4 v = *reinterpret_cast<const int4*>(kb + tt * D * 2 + (sub + j * LPT) * 16);
        bf16x8_to_f32(v, kf + j * 8);
      }
      float d[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float2 a = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < EL; e += 2)
          a = __ffma2_rn(make_float2(qr[r][e], qr[r][e + 1]), make_float2(kf[e], kf[e + 1]), a);
        d[r] = a.x + a.y;
      }
      reduce_scatter<R, LPT / 2>(d, lane);
      float sv = d[0];
      if (!fast) {
        const int pos = pos0 + tt;
        if (pos >= task.kv_end || pos > my_lim) sv = -INFINITY;
      }
      sc[it] = sv;
    }
    if (TREE && !fast) {                       // warp-uniform; kept out of the loop above
#pragma unroll
      for (int it = 0; it < ITERS; ++it) {
        const int back = my_lim - (pos0 + it * TPW + grp);
        if (back >= 0 && back < 64 && !((my_mask >> back) & 1ull)) sc[it] = -INFINITY;
      }
    }
    float mx = sc[0];
#pragma unroll
    for (int it = 1; it < ITERS; ++it) mx = fmaxf(mx, sc[it]);
#pragma unroll
    for (int o = LPT; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const bool need = (mx > m_run + 8.f) || (m_run == -INFINITY && mx != -INFINITY);
    if (__any_sync(0xffffffffu, need)) {
      const float m_new = need ? fmaxf(mx, m_run) : m_run;
      const float alpha = (m_run == -INFINITY) ? 0.f : fast_ex2(m_run - m_new);
      m_run = m_new;
      l_run *= alpha;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float a = __shfl_sync(0xffffffffu, alpha, rs_lane<R, LPT>(r));
#pragma unroll
        for (int e = 0; e < EL; ++e) acc[r][e] *= a;
      }
    }
    const float msub = (m_run == -INFINITY) ? 0.f : m_run;
    float ls = 0.f;
#pragma unroll
    for (int it = 0; it < ITERS; ++it) {
      sc[it] = fast_ex2(sc[it] - msub);
      ls += sc[it];
    }
#pragma unroll
    for (int o = LPT; o < 32; o <<= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
    l_run += ls;
#pragma unroll
    for (int it = 0; it < ITERS; ++it) {
      const int tt = it * TPW + grp;
      float vf[EL];
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        const int4 v = *reinterpret_cast<const int4*>(vb + tt * D * 2 + (sub + j * LPT) * 16);
        bf16x8_to_f32(v, vf + j * 8);
      }
      if (!fast && pos0 + tt >= task.kv_end) {
#pragma unroll
        for (int e = 0; e < EL; ++e) vf[e] = 0.f;   // rows past the end may hold NaN
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float pr = __shfl_sync(0xffffffffu, sc[it], grp * LPT + rs_lane<R, LPT>(r));
#pragma unroll
        for (int e = 0; e < EL; e += 2) {
          const float2 o2 = __ffma2_rn(make_float2(pr, pr), make_float2(vf[e], vf[e + 1]),
                                       make_float2(acc[r][e], acc[r][e + 1]));
          acc[r][e] = o2.x;
          acc[r][e + 1] = o2.y;
        }
      }
    }
    __syncwarp();
    if (lane == 0) sm100::mbar_arrive(sm100::smem_u32(&sh.empty[s]));
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int e = 0; e < EL; ++e)
#pragma unroll
      for (int o = LPT; o < 32; o <<= 1) acc[r][e] += __shfl_xor_sync(0xffffffffu, acc[r][e], o);

  // The previous task's combine readers are done (consumer warps only; the
  // producer keeps streaming the next task meanwhile), then write this warp's
  // state.  Rows R..RS-1 of the buffer are unused for this task.
  asm volatile("bar.sync 1, %0;" ::"r"(kBw2Consumers * 32) : "memory");
  if (grp == 0) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int j = 0; j < CH; ++j)
#pragma unroll
        for (int x = 0; x < 8; ++x)
          sh.co[(warp * RS + r) * D + (sub + j * LPT) * 8 + x] = acc[r][j * 8 + x];
    if (lane == rs_lane<R, LPT>(my_row)) {
      sh.cm[warp * RS + my_row] = m_run;
      sh.cl[warp * RS + my_row] = l_run;
    }
  }
  return live;
}

// TREE: the batch holds draft-tree verify rows (per-token lookback masks);
// batches without one run the TREE = false instance, which has no mask code.
template <int D, int R, bool TREE>
__global__ void __launch_bounds__(kBw2Threads, 1) bw2_attention_kernel(
    const pps::Task* __restrict__ tasks, int32_t num_tasks, const int32_t* __restrict__ rows,
    const int32_t* __restrict__ pages, const __nv_bfloat16* __restrict__ q,
    const __nv_bfloat16* __restrict__ pool_k, const __nv_bfloat16* __restrict__ pool_v,
    __nv_bfloat16* __restrict__ out, float* __restrict__ o_part, float* __restrict__ lse_part,
    const unsigned long long* __restrict__ tree_mask, int32_t* __restrict__ err,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t G, int32_t page_size, float qk_scale) {
  using C = Bw2<D, R>;
  using S = Bw3Smem<D, R>;
  extern __shared__ __align__(128) uint8_t bw2_smem[];
  __shared__ uint64_t full[kBw2Stages], empty[kBw2Stages], qfull[2], qempty[2];
  __shared__ volatile int abort_flag;
  // Per task (double-buffered with the query rows): the task record and its
  // token ids, written by the producer so consumers never wait on global loads.
  __shared__ pps::Task tinfo[2];
  __shared__ int32_t ttok[2][R];
  __shared__ unsigned long long tmsk[2][R];   // draft-tree lookback mask per token

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x, nctas = gridDim.x;
  if (tid == 0) {
    for (int s = 0; s < kBw2Stages; ++s) {
      sm100::mbar_init(sm100::smem_u32(&full[s]), 1);
      sm100::mbar_init(sm100::smem_u32(&empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      sm100::mbar_init(sm100::smem_u32(&qfull[i]), 1);
      sm100::mbar_init(sm100::smem_u32(&qempty[i]), kBw2Consumers);
    }
    abort_flag = 0;
    sm100::fence_mbar_init();
  }
  __syncthreads();
  // Set-up done: let the next kernel of the stream be scheduled, then wait
  // for the one before (the append writes the pool rows this kernel reads).
  sm100::grid_dep_launch();
  sm100::grid_dep_wait();
  auto fail = [&]() {
    atomicCAS(err, 0, PPS_DEV_ERR_WAIT_TIMEOUT);
    abort_flag = 1;
  };

  if (warp == kBw2Consumers) {
    // ---------------------------------------------------------------- producer
    // The whole warp walks the CTA's tasks: lanes fetch 32 page ids at a time
    // (one coalesced load instead of a dependent load per sub-block) and lane 0
    // issues the bulk copies.
    const size_t head_stride = (size_t)page_size * D;
    const uint32_t half = kBw2Sub * D * 2;
    int gk = 0, t;
    bool ok = true;
    for (int ti = 0; ok && (t = snake_task(ti, b, nctas)) < num_tasks; ++ti) {
      const pps::Task task = tasks[t];
      const int qb = ti & 1, quse = ti >> 1;
      if (lane == 0) {
        ok = !(quse > 0 && !sm100::mbar_wait(sm100::smem_u32(&qempty[qb]), (quse - 1) & 1)) &&
             !abort_flag;
        if (ok) {
          tinfo[qb] = task;
          for (int i = 0; i < task.n_tok; ++i) {
            ttok[qb][i] = rows[task.row_off + i];
            if constexpr (TREE)
              tmsk[qb][i] = task.causal != PPS_NO_CAUSAL ? tree_mask[ttok[qb][i]] : ~0ull;
          }
          const uint32_t qbar = sm100::smem_u32(&qfull[qb]);
          const uint32_t tok_bytes = (uint32_t)G * D * 2;
          sm100::mbar_expect_tx(qbar, tok_bytes * task.n_tok);   // releases tinfo / ttok
          for (int i = 0; i < task.n_tok; ++i)
            bulk_g2s(sm100::smem_u32(bw2_smem + S::qbuf + qb * ((S::qbuf_bytes + 127) / 128 * 128)) +
                         i * tok_bytes,
                     q + ((size_t)ttok[qb][i] * num_q_heads + task.kv_head * G) * D, tok_bytes,
                     qbar);
        } else {
          fail();
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      // K/V sub-blocks in batches of kIssueLanes: lane j loads the page id of
      // sub-block k0 + j, waits for its ring stage and issues its two copies.
      // A single issuing thread cannot keep 4 KB copies in flight fast enough
      // to saturate HBM; several lanes issuing at once can.
      const int n_sub = (task.kv_end - task.kv_begin + kBw2Sub - 1) / kBw2Sub;
      for (int k0 = 0; ok && k0 < n_sub; k0 += kIssueLanes) {
        const int cnt = min(kIssueLanes, n_sub - k0);
        bool good = true;
        if (lane < cnt) {
          const int g = gk + k0 + lane;
          const int wi = g / kBw2Consumers;                 // index within its warp's stream
          const int st = (g % kBw2Consumers) * kStagesPerWarp + wi % kStagesPerWarp;
          const int use = wi / kStagesPerWarp;
          const int pos0 = task.kv_begin + (k0 + lane) * kBw2Sub;
          const int page = pages[task.page_off + pos0 / page_size];
          if (use > 0 && !sm100::mbar_wait(sm100::smem_u32(&empty[st]), (use - 1) & 1)) {
            good = false;
          } else if (abort_flag) {
            good = false;
          } else {
            const size_t off = ((size_t)page * num_kv_heads + task.kv_head) * head_stride +
                               (size_t)(pos0 % page_size) * D;
            const uint32_t bar = sm100::smem_u32(&full[st]);
            const uint32_t dst = sm100::smem_u32(bw2_smem + S::ring + st * C::STAGE);
            sm100::mbar_expect_tx(bar, 2 * half);
            bulk_g2s(dst, pool_k + off, half, bar);
            bulk_g2s(dst + half, pool_v + off, half, bar);
          }
          if (!good) fail();
        }
        ok = __all_sync(0xffffffffu, good);
      }
      gk += n_sub;
    }
    // every started copy lands before the CTA may exit (after a failed wait
    // some of the last stages were never armed: short bounded waits there)
    if (lane == 0) {
      for (int g = (gk > kBw2Stages ? gk - kBw2Stages : 0); g < gk; ++g) {
        const int wi = g / kBw2Consumers;
        const int st = (g % kBw2Consumers) * kStagesPerWarp + wi % kStagesPerWarp;
        sm100::mbar_wait(sm100::smem_u32(&full[st]), (wi / kStagesPerWarp) & 1,
                         ok ? 2000000000ull : 10000000ull);
      }
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  float* cm = reinterpret_cast<float*>(bw2_smem + S::comb);   // [warps][R] max
  float* cl = cm + kBw2Consumers * R;                          // [warps][R] sum
  float* co = cl + kBw2Consumers * R;                          // [warps][R][D]
  BwShared sh{bw2_smem + S::ring, full, empty, &abort_flag, err, cm, cl, co};
  int gk = 0, t;
  for (int ti = 0; (t = snake_task(ti, b, nctas)) < num_tasks; ++ti) {
    bool live = !abort_flag;
    // task record, token ids and query rows from the producer's buffers
    const int qb = ti & 1;
    if (live) {
      const bool got = sm100::mbar_wait(sm100::smem_u32(&qfull[qb]), (ti >> 1) & 1);
      if (!__all_sync(0xffffffffu, got)) { if (lane == 0) fail(); live = false; }
    }
    const pps::Task task = live ? tinfo[qb] : tasks[t];
    int32_t tok[R];
#pragma unroll
    for (int i = 0; i < R; ++i) tok[i] = (live && i < task.n_tok) ? ttok[qb][i] : 0;
    const int nrows = task.n_tok * G;
    const int n_sub = (task.kv_end - task.kv_begin + kBw2Sub - 1) / kBw2Sub;
    const uint8_t* qs = bw2_smem + S::qbuf + qb * ((S::qbuf_bytes + 127) / 128 * 128);
    // Tasks of up to 4 rows (one decode token at G = 4) take the 4-row inner
    // loop even in the 8-row instance: half the arithmetic per K/V byte.
    if (R == 8 && nrows <= 4)
      live = bw_consume<D, (R == 8 ? 4 : R), R, TREE>(task, nrows, G, n_sub, gk, qs, tmsk[qb],
                                                       qk_scale, live, sh, &qempty[qb]);
    else
      live = bw_consume<D, R, R, TREE>(task, nrows, G, n_sub, gk, qs, tmsk[qb], qk_scale, live,
                                       sh, &qempty[qb]);
    gk += n_sub;
    asm volatile("bar.sync 1, %0;" ::"r"(kBw2Consumers * 32) : "memory");
    for (int idx = tid; idx < nrows * D; idx += kBw2Consumers * 32) {
      const int r = idx / D, c = idx - (idx / D) * D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kBw2Consumers; ++w) M = fmaxf(M, cm[w * R + r]);
      float o = 0.f, l = 0.f;
#pragma unroll
      for (int w = 0; w < kBw2Consumers; ++w) {
        const float mw = cm[w * R + r];
        const float sw = (mw == -INFINITY) ? 0.f : fast_ex2(mw - M);
        o += sw * co[(w * R + r) * D + c];
        l += sw * cl[w * R + r];
      }
      const float val = l > 0.f ? o / l : 0.f;
      const int i = r / G, h = task.kv_head * G + r % G;
      if (!live) continue;
      int ti_tok = tok[0];
#pragma unroll
      for (int x = 1; x < R; ++x) if (x == i) ti_tok = tok[x];
      if (task.out_pid < 0) {
        out[((size_t)ti_tok * num_q_heads + h) * D + c] = __float2bfloat16_rn(val);
      } else {
        const size_t prow = (size_t)(task.out_pid + i) * num_q_heads + h;
        o_part[prow * D + c] = val;
        if (c == 0) lse_part[prow] = l > 0.f ? M + log2f(l) : -INFINITY;
      }
    }
  }
}

template <int D, int R, bool TREE>
int launch_v2(const pps::Shape& s, const pps::DeviceTables& t, int64_t n, const void* q,
              const pps_pool& pool, void* out, int32_t* err, cudaStream_t st) {
  auto kern = bw2_attention_kernel<D, R, TREE>;
  constexpr int smem = Bw3Smem<D, R>::total;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return (int)e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return (int)e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return (int)e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kBw2Threads, smem)) !=
      cudaSuccess)
    return (int)e;
  const int64_t grid = std::min<int64_t>(n, (int64_t)sms * std::max(per_sm, 1));
  e = pps::launch_dependent(
      kern, (unsigned)grid, kBw2Threads, smem, st, (const pps::Task*)t.bw_tasks, (int32_t)n,
      (const int32_t*)t.rows, (const int32_t*)t.pages, (const __nv_bfloat16*)q,
      (const __nv_bfloat16*)pool.k, (const __nv_bfloat16*)pool.v, (__nv_bfloat16*)out, t.o_part,
      t.lse_part, t.tree_mask, err, s.num_q_heads, s.num_kv_heads, s.group, s.page_size,
      s.sm_scale * kLog2e);
  pps::count_launch();
  return (int)e;
}

template <int D, int R>
int launch_t(const pps::Shape& s, const pps::DeviceTables& t, int64_t n, const void* q,
             const pps_pool& pool, void* out, cudaStream_t st) {
  const size_t score_bytes = (size_t)R * kKB * 4;
  const size_t red_bytes = (size_t)4 * R * D * 4;
  const size_t smem = (size_t)4 * R * 4 + (score_bytes > red_bytes ? score_bytes : red_bytes);
  auto kern = bw_attention_kernel<D, R>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
  }
  kern<<<(unsigned)n, kThreads, smem, st>>>(
      t.bw_tasks, t.rows, t.pages, (const __nv_bfloat16*)q, (const __nv_bfloat16*)pool.k,
      (const __nv_bfloat16*)pool.v, (__nv_bfloat16*)out, t.o_part, t.lse_part, t.tree_mask,
      s.num_q_heads, s.num_kv_heads, s.group, s.page_size, s.sm_scale * kLog2e);
  pps::count_launch();
  return (int)cudaGetLastError();
}

}  // namespace

namespace pps {

int launch_bw_attention(const Shape& s, const DeviceTables& t, int64_t num_tasks, const void* q,
                        const pps_pool& pool, void* out, int32_t* err, void* stream,
                        const AppendArgs* app) {
  if (num_tasks == 0) return cudaSuccess;
  if (s.small_tt) return launch_tt_attention(s, t, num_tasks, q, pool, out, err, stream, app);
  if (app) return (int)cudaErrorInvalidValue;        // the CUDA-core kernels do not append
  auto st = (cudaStream_t)stream;
  // The planner caps rows per task at kBwMaxRows; pick the smallest instance.
  // Up to 8 rows: the pipelined v2 kernel; 9..16 rows (CUDA-core-only plans): v1.
  const int rows = s.bw_rows_max;
  const bool tree = t.tree_mask != nullptr;
  if (s.head_dim == 128) {
    if (rows <= 4) return tree ? launch_v2<128, 4, true>(s, t, num_tasks, q, pool, out, err, st)
                               : launch_v2<128, 4, false>(s, t, num_tasks, q, pool, out, err, st);
    if (rows <= 8) return tree ? launch_v2<128, 8, true>(s, t, num_tasks, q, pool, out, err, st)
                               : launch_v2<128, 8, false>(s, t, num_tasks, q, pool, out, err, st);
    return launch_t<128, 16>(s, t, num_tasks, q, pool, out, st);
  }
  if (rows <= 4) return tree ? launch_v2<64, 4, true>(s, t, num_tasks, q, pool, out, err, st)
                             : launch_v2<64, 4, false>(s, t, num_tasks, q, pool, out, err, st);
  if (rows <= 8) return tree ? launch_v2<64, 8, true>(s, t, num_tasks, q, pool, out, err, st)
                             : launch_v2<64, 8, false>(s, t, num_tasks, q, pool, out, err, st);
  return launch_t<64, 16>(s, t, num_tasks, q, pool, out, st);
}

}  // namespace pps
