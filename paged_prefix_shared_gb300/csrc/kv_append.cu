// kv_append: scatter this step's new K/V rows into their pool pages.
//
// Definition: PagedAttention block table (XY-Serve review, "Assumptions & free
// parameters"); new token j of request r is written at logical position
// cached_len[r] + j, i.e. page page_indices[page_indptr[r] + p / P], slot p % P.
//
// One warp per (token, kv head): lanes copy the head_dim-long K row and V row
// with 16-byte vector loads/stores (head_dim 128 -> 16 lanes per row, K and V
// in the two half-warps).  Pure data movement: bit exact by construction.
#include <cuda_runtime.h>

#include "pps_internal.h"
#include "sm100_ptx.cuh"
#include "append_dev.cuh"

namespace {

__device__ __forceinline__ void set_error(int32_t* err, int32_t code) {
  atomicCAS(err, 0, code);
}

template <int D>
__global__ void __launch_bounds__(256) kv_append_kernel(
    int4* __restrict__ pool_k, int4* __restrict__ pool_v, const int4* __restrict__ k_new,
    const int4* __restrict__ v_new, const int32_t* __restrict__ q_indptr,
    const int32_t* __restrict__ cached_len, const int32_t* __restrict__ page_indptr,
    const int32_t* __restrict__ page_indices, int32_t num_requests, int32_t num_tokens,
    int32_t num_kv_heads, int32_t page_size, int32_t num_pages, int32_t* __restrict__ err) {
  constexpr int kVec = D * 2 / 16;                  // int4 per row (8 or 16)
  // the attention kernels that follow may be scheduled now (they wait for
  // this grid's writes before reading the pool)
  sm100::grid_dep_launch();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int t = warp / num_kv_heads;
  const int h = warp - t * num_kv_heads;
  if (t >= num_tokens) return;
  // request of token t: last r with q_indptr[r] <= t
  if (q_indptr[0] > t || q_indptr[num_requests] <= t) {
    if (lane == 0) set_error(err, PPS_DEV_ERR_APPEND_REQUEST);
    return;
  }
  const int r = pps_dev::request_of_token(q_indptr, num_requests, t, lane);
  const int p = cached_len[r] + (t - q_indptr[r]);
  const int pi = p / page_size;
  const int npg = page_indptr[r + 1] - page_indptr[r];
  if (p < 0 || pi >= npg) {
    if (lane == 0) set_error(err, PPS_DEV_ERR_APPEND_PAGE_LIST);
    return;
  }
  const int page = page_indices[page_indptr[r] + pi];
  if (page < 0 || page >= num_pages) {
    if (lane == 0) set_error(err, PPS_DEV_ERR_APPEND_PAGE_ID);
    return;
  }
  const int slot = p - pi * page_size;
  const size_t dst = (((size_t)page * num_kv_heads + h) * page_size + slot) * kVec;
  const size_t src = ((size_t)t * num_kv_heads + h) * kVec;
  if (kVec == 16) {
    if (lane < 16) pool_k[dst + lane] = __ldg(k_new + src + lane);
    else pool_v[dst + lane - 16] = __ldg(v_new + src + lane - 16);
  } else {
    if (lane < kVec) pool_k[dst + lane] = __ldg(k_new + src + lane);
    else if (lane < 2 * kVec) pool_v[dst + lane - kVec] = __ldg(v_new + src + lane - kVec);
  }
}

// The same scatter with each new token's (page, slot) computed on the host from
// the step's checked tables (the step calls): one warp per (token, kv head),
// one dependent load before the copy instead of a request search and two
// table lookups.
template <int D>
__global__ void __launch_bounds__(256) kv_append_slots_kernel(
    int4* __restrict__ pool_k, int4* __restrict__ pool_v, const int4* __restrict__ k_new,
    const int4* __restrict__ v_new, const int2* __restrict__ dst_slots, int32_t num_tokens,
    int32_t num_kv_heads, int32_t page_size) {
  constexpr int kVec = D * 2 / 16;
  sm100::grid_dep_launch();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int t = warp / num_kv_heads;
  const int h = warp - t * num_kv_heads;
  if (t >= num_tokens) return;
  const int2 ps = __ldg(dst_slots + t);              // {page, slot}
  const size_t dst = (((size_t)ps.x * num_kv_heads + h) * page_size + ps.y) * kVec;
  const size_t src = ((size_t)t * num_kv_heads + h) * kVec;
  if (lane < kVec) pool_k[dst + lane] = __ldg(k_new + src + lane);
  else if (lane < 2 * kVec) pool_v[dst + lane - kVec] = __ldg(v_new + src + lane - kVec);
}

// Copy-on-write of a partly reused page: slots [0, n) of every kv head of page
// src go to the same slots of page dst (K and V), one warp per (copy, kv head,
// slot).  A page id out of range or a slot count outside [0, page_size] is
// skipped and recorded in the device error word.
template <int D>
__global__ void __launch_bounds__(256) copy_slots_kernel(
    int4* __restrict__ pool_k, int4* __restrict__ pool_v, const int32_t* __restrict__ src_pages,
    const int32_t* __restrict__ dst_pages, const int32_t* __restrict__ num_slots, int32_t count,
    int32_t num_kv_heads, int32_t page_size, int32_t num_pages, int32_t* __restrict__ err) {
  constexpr int kVec = D * 2 / 16;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t per_copy = (int64_t)num_kv_heads * page_size;
  const int64_t c = warp / per_copy;
  if (c >= count) return;
  const int rem = (int)(warp - c * per_copy);
  const int h = rem / page_size, slot = rem - h * page_size;
  const int src = src_pages[c], dst = dst_pages[c], n = num_slots[c];
  if (src < 0 || src >= num_pages || dst < 0 || dst >= num_pages || n < 0 || n > page_size) {
    if (lane == 0 && h == 0 && slot == 0) set_error(err, PPS_DEV_ERR_COPY_ARGUMENT);
    return;
  }
  if (slot >= n) return;
  const size_t so = (((size_t)src * num_kv_heads + h) * page_size + slot) * kVec;
  const size_t d0 = (((size_t)dst * num_kv_heads + h) * page_size + slot) * kVec;
  if (lane < kVec) pool_k[d0 + lane] = pool_k[so + lane];
  else if (lane < 2 * kVec) pool_v[d0 + lane - kVec] = pool_v[so + lane - kVec];
}

}  // namespace

namespace pps {

int launch_copy_slots(const pps_pool& pool, const int32_t* src_pages, const int32_t* dst_pages,
                      const int32_t* num_slots, int32_t count, int32_t* err, void* stream) {
  const int64_t warps = (int64_t)count * pool.num_kv_heads * pool.page_size;
  if (warps == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (warps * 32 + threads - 1) / threads;
  auto s = (cudaStream_t)stream;
  if (pool.head_dim == 128)
    copy_slots_kernel<128><<<(unsigned)blocks, threads, 0, s>>>(
        (int4*)pool.k, (int4*)pool.v, src_pages, dst_pages, num_slots, count, pool.num_kv_heads,
        pool.page_size, pool.num_pages, err);
  else
    copy_slots_kernel<64><<<(unsigned)blocks, threads, 0, s>>>(
        (int4*)pool.k, (int4*)pool.v, src_pages, dst_pages, num_slots, count, pool.num_kv_heads,
        pool.page_size, pool.num_pages, err);
  count_launch();
  return (int)cudaGetLastError();
}

int launch_kv_append_slots(const pps_pool& pool, const void* k_new, const void* v_new,
                           const int32_t* dst_slots, int32_t num_new_tokens, void* stream) {
  const int64_t warps = (int64_t)num_new_tokens * pool.num_kv_heads;
  if (warps == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (warps * 32 + threads - 1) / threads;
  auto s = (cudaStream_t)stream;
  auto kern = pool.head_dim == 128 ? kv_append_slots_kernel<128> : kv_append_slots_kernel<64>;
  kern<<<(unsigned)blocks, threads, 0, s>>>((int4*)pool.k, (int4*)pool.v, (const int4*)k_new,
                                            (const int4*)v_new,
                                            reinterpret_cast<const int2*>(dst_slots),
                                            num_new_tokens, pool.num_kv_heads, pool.page_size);
  count_launch();
  return (int)cudaGetLastError();
}

int launch_kv_append(const pps_pool& pool, const void* k_new, const void* v_new,
                     const int32_t* q_indptr, const int32_t* cached_len,
                     const int32_t* page_indptr, const int32_t* page_indices,
                     int32_t num_requests, int32_t num_new_tokens, int32_t* err, void* stream) {
  const int64_t warps = (int64_t)num_new_tokens * pool.num_kv_heads;
  if (warps == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (warps * 32 + threads - 1) / threads;
  auto s = (cudaStream_t)stream;
  if (pool.head_dim == 128)
    kv_append_kernel<128><<<(unsigned)blocks, threads, 0, s>>>(
        (int4*)pool.k, (int4*)pool.v, (const int4*)k_new, (const int4*)v_new, q_indptr,
        cached_len, page_indptr, page_indices, num_requests, num_new_tokens, pool.num_kv_heads,
        pool.page_size, pool.num_pages, err);
  else
    kv_append_kernel<64><<<(unsigned)blocks, threads, 0, s>>>(
        (int4*)pool.k, (int4*)pool.v, (const int4*)k_new, (const int4*)v_new, q_indptr,
        cached_len, page_indptr, page_indices, num_requests, num_new_tokens, pool.num_kv_heads,
        pool.page_size, pool.num_pages, err);
  count_launch();
  return (int)cudaGetLastError();
}

}  // namespace pps
