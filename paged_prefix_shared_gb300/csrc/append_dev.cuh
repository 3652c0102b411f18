// The step's K/V append done inside an attention kernel's set-up (the
// kv_append launch fused into the attention launch).
//
// Every CTA of the (cooperatively launched, so all resident) kernel copies a
// share of the new rows into their pool pages -- the same copy as
// pps_kv_append: new token j of request r goes to logical position
// cached_len[r] + j, page page_indices[page_indptr[r] + p / P], slot p % P
// (XY-Serve review, "Assumptions & free parameters": the paged block table) --
// then all CTAs wait for one another on a counter before any task reads the
// pool.  The wait is bounded: if it runs out, the kernel records
// PPS_DEV_ERR_WAIT_TIMEOUT and goes on.
#pragma once

#include <cstdint>

#include "pps_internal.h"

namespace pps_dev {

// The request of new token t, the last r with q_indptr[r] <= t (empty requests
// have equal consecutive offsets, so this is the one that holds t), found by a
// whole warp: each round its 32 lanes probe 32 evenly spaced offsets at once
// and the range shrinks 32-fold, so a 256-request batch takes 2 dependent
// loads instead of the 8 of a one-thread bisection.  The caller has checked
// q_indptr[0] <= t < q_indptr[num_requests]; every lane gets the answer.
__device__ __forceinline__ int request_of_token(const int32_t* q_indptr, int num_requests,
                                                int t, int lane) {
  int lo = 0, hi = num_requests;                    // q_indptr[lo] <= t < q_indptr[hi]
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) >> 5;
    const int probe = lo + (lane + 1) * step;
    const bool le = probe < hi && __ldg(q_indptr + probe) <= t;
    const int c = __popc(__ballot_sync(0xffffffffu, le));   // probes <= t: a prefix of lanes
    hi = min(hi, lo + (c + 1) * step);
    lo += c * step;
  }
  return lo;
}

// One warp per (new token, kv head) item, items strided over every warp of the
// grid; the caller's `nwarps` warps of this CTA take part (warps 0..nwarps-1).
template <int D>
__device__ __noinline__ void append_rows(const pps::AppendArgs& a, int4* pool_k, int4* pool_v,
                                            int32_t num_kv_heads, int32_t page_size,
                                            int32_t num_pages, int32_t* err, int warp, int lane,
                                            int nwarps) {
  constexpr int kVec = D * 2 / 16;                   // int4 per row (8 or 16)
  const int64_t items = (int64_t)a.num_tokens * num_kv_heads;
  const int64_t stride = (int64_t)gridDim.x * nwarps;
  const int4* k_new = reinterpret_cast<const int4*>(a.k_new);
  const int4* v_new = reinterpret_cast<const int4*>(a.v_new);
  for (int64_t w = (int64_t)blockIdx.x * nwarps + warp; w < items; w += stride) {
    const int t = (int)(w / num_kv_heads);
    const int h = (int)(w - (int64_t)t * num_kv_heads);
    if (a.q_indptr[0] > t || a.q_indptr[a.num_requests] <= t) {
      if (lane == 0) atomicCAS(err, 0, PPS_DEV_ERR_APPEND_REQUEST);
      continue;
    }
    const int r = request_of_token(a.q_indptr, a.num_requests, t, lane);
    const int p = a.cached_len[r] + (t - a.q_indptr[r]);
    const int pi = p / page_size;
    if (p < 0 || pi >= a.page_indptr[r + 1] - a.page_indptr[r]) {
      if (lane == 0) atomicCAS(err, 0, PPS_DEV_ERR_APPEND_PAGE_LIST);
      continue;
    }
    const int page = a.page_indices[a.page_indptr[r] + pi];
    if (page < 0 || page >= num_pages) {
      if (lane == 0) atomicCAS(err, 0, PPS_DEV_ERR_APPEND_PAGE_ID);
      continue;
    }
    const size_t dst = (((size_t)page * num_kv_heads + h) * page_size + (p - pi * page_size)) * kVec;
    const size_t src = ((size_t)t * num_kv_heads + h) * kVec;
    if (lane < kVec) pool_k[dst + lane] = k_new[src + lane];
    else if (lane < 2 * kVec) pool_v[dst + lane - kVec] = v_new[src + lane - kVec];
  }
  // these generic-proxy writes are read by TMA / bulk copies (async proxy)
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Every CTA of the grid arrives once; returns when all have (or after about a
// second, recording the timeout).  Called by every thread of the CTA.
static __device__ __noinline__ void grid_wait(int32_t* counter, int32_t* err) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(counter, 1);
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    while (true) {
      int32_t seen;
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(seen) : "l"(counter) : "memory");
      if (seen >= (int32_t)gridDim.x) break;
      uint64_t t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > 1000000000ull) {
        atomicCAS(err, 0, PPS_DEV_ERR_WAIT_TIMEOUT);
        break;
      }
      __nanosleep(100);
    }
    __threadfence();
  }
  __syncthreads();
}

}  // namespace pps_dev
