// Partial-softmax merge: combine the (o_i, lse_i) partials of every split
// (token, query head) into the final bf16 output row.
//
// With M = max_i lse_i (log2 domain) the merged row is
//   sum_i 2^(lse_i - M) o_i / sum_i 2^(lse_i - M),
// o_i being already normalised by its own softmax sum.  This is the split the
// online-softmax equivalence allows (XY-Serve review, "Assumptions & free
// parameters"; Flash-Decoding in its reference list).  A partial whose rows
// saw no key has lse = -inf and weight 0.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "pps_internal.h"
#include "sm100_ptx.cuh"

namespace {

// One warp per (merged token, query head); each lane owns D/32 consecutive
// output columns.  Enough independent warps to cover the memory latency of
// the few partial rows each one reads.
template <int D>
__global__ void __launch_bounds__(256) merge_kernel(
    const int32_t* __restrict__ tokens, const int32_t* __restrict__ indptr,
    const int32_t* __restrict__ pids, const float* __restrict__ o_part,
    const float* __restrict__ lse_part, __nv_bfloat16* __restrict__ out, int32_t num_q_heads,
    int64_t num_rows) {
  constexpr int kPer = D / 32;
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const bool live = wid < num_rows;
  const int m = live ? (int)(wid / num_q_heads) : 0;
  const int h = live ? (int)(wid - (int64_t)m * num_q_heads) : 0;
  // The merge lists were uploaded before the step's kernels ran, so they are
  // read while the attention kernel before this one finishes; only the
  // partials wait for it.
  // (the first three partial ids are read ahead; a token rarely has more)
  int t = 0, a = 0, b = 0, p0 = 0, p1 = 0, p2 = 0;
  if (live) {
    t = __ldg(tokens + m);
    a = __ldg(indptr + m);
    b = __ldg(indptr + m + 1);
    if (a < b) p0 = __ldg(pids + a);
    if (a + 1 < b) p1 = __ldg(pids + a + 1);
    if (a + 2 < b) p2 = __ldg(pids + a + 2);
  }
  sm100::grid_dep_wait();        // the partials of the attention kernels before it
  if (!live) return;
  auto pid_at = [&](int i) {
    const int d = i - a;
    return d == 0 ? p0 : d == 1 ? p1 : d == 2 ? p2 : __ldg(pids + i);
  };
  float M = -INFINITY;
  for (int i = a; i < b; ++i) M = fmaxf(M, lse_part[(size_t)pid_at(i) * num_q_heads + h]);
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  for (int i = a; i < b; ++i) {
    const size_t row = (size_t)pid_at(i) * num_q_heads + h;
    const float l = lse_part[row];
    const float w = (l == -INFINITY) ? 0.f : exp2f(l - M);
    wsum += w;
    const float* src = o_part + row * D + lane * kPer;
    if constexpr (kPer == 4) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      acc[0] += w * v.x; acc[1] += w * v.y; acc[2] += w * v.z; acc[3] += w * v.w;
    } else {
      static_assert(kPer == 2, "head_dim 64 or 128");
      const float2 v = *reinterpret_cast<const float2*>(src);
      acc[0] += w * v.x; acc[1] += w * v.y;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat16* dst = out + ((size_t)t * num_q_heads + h) * D + lane * kPer;
#pragma unroll
  for (int e = 0; e < kPer; e += 2)
    *reinterpret_cast<__nv_bfloat162*>(dst + e) = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
}

}  // namespace

namespace pps {

int launch_merge(const Shape& s, const DeviceTables& t, int64_t num_merge_tokens, void* out,
                 void* stream) {
  if (num_merge_tokens == 0) return cudaSuccess;
  auto st = (cudaStream_t)stream;
  const int64_t rows = num_merge_tokens * s.num_q_heads;
  const unsigned blocks = (unsigned)((rows * 32 + 255) / 256);
  auto kern = s.head_dim == 128 ? merge_kernel<128> : merge_kernel<64>;
  const cudaError_t e = launch_dependent(
      kern, blocks, 256, 0, st, (const int32_t*)t.merge_tokens, (const int32_t*)t.merge_indptr,
      (const int32_t*)t.merge_pids, (const float*)t.o_part, (const float*)t.lse_part,
      (__nv_bfloat16*)out, s.num_q_heads, rows);
  count_launch();
  return (int)e;
}

}  // namespace pps
