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
#include <cuda_runtime.h>

#include "pps_internal.h"

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
    int32_t num_q_heads, int32_t num_kv_heads, int32_t G, int32_t page_size, float qk_scale) {
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
          const bool vis = p <= task.causal + r / G;
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
      (const __nv_bfloat16*)pool.v, (__nv_bfloat16*)out, t.o_part, t.lse_part, s.num_q_heads,
      s.num_kv_heads, s.group, s.page_size, s.sm_scale * kLog2e);
  pps::count_launch();
  return (int)cudaGetLastError();
}

}  // namespace

namespace pps {

int launch_bw_attention(const Shape& s, const DeviceTables& t, int64_t num_tasks, const void* q,
                        const pps_pool& pool, void* out, int32_t* /*err*/, void* stream) {
  if (num_tasks == 0) return cudaSuccess;
  auto st = (cudaStream_t)stream;
  // The planner caps rows per task at kBwMaxRows; pick the smallest instance.
  const int rows = s.bw_rows_max;
  if (s.head_dim == 128) {
    if (rows <= 4) return launch_t<128, 4>(s, t, num_tasks, q, pool, out, st);
    if (rows <= 8) return launch_t<128, 8>(s, t, num_tasks, q, pool, out, st);
    return launch_t<128, 16>(s, t, num_tasks, q, pool, out, st);
  }
  if (rows <= 4) return launch_t<64, 4>(s, t, num_tasks, q, pool, out, st);
  if (rows <= 8) return launch_t<64, 8>(s, t, num_tasks, q, pool, out, st);
  return launch_t<64, 16>(s, t, num_tasks, q, pool, out, st);
}

}  // namespace pps
