// Virtual-padded projection GEMM (pps_gemm_bf16): C = A W^T for the token rows
// of a mixed batch, A [M, K], W [N, K], C [M, N], all bf16 row-major, M any.
//
// XY-Serve review (pith.science/paper/ABCKJ6RF), "Core claim": SmoothGEMM
// keeps the efficiency of fixed-shape kernels for arbitrary shapes by padding
// virtually in on-chip buffers and reading/writing only real data.  Here the
// fixed shape is a 128 x 256 output tile; TMA loads of a tile that runs past
// M, N or K fill the out-of-range part of the shared-memory tile with zeros
// (the virtual padding), nothing padded is ever read from or written to HBM,
// and the epilogue stores only rows < M and columns < N.
//
// Persistent kernel, one CTA per SM (192 threads) taking output tiles b,
// b + grid, ...:
//   warp 0     TMA producer: per 64-wide K block, the A tile (128 x 64) and the
//              W tile (256 x 64), 128-byte swizzle, into a 4-stage ring;
//   warp 1     MMA issuer: 4 x tcgen05.mma (M 128, N 256, K 16) per K block into
//              one of two TMEM accumulators (2 x 256 columns), so the epilogue
//              of one tile overlaps the MMAs of the next;
//   warps 2-5  epilogue: TMEM -> registers -> bf16 -> global, row = TMEM lane.
// Every mbarrier wait is bounded; on timeout the kernel records
// PPS_DEV_ERR_WAIT_TIMEOUT, stops, drains what it issued and frees TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "pps_internal.h"
#include "sm100_ptx.cuh"

namespace {

using namespace sm100;

constexpr int kBM = 128, kBN = 256, kBK = 64, kStages = 4;
constexpr int kABytes = kBM * kBK * 2;              // 16 KB
constexpr int kBBytes = kBN * kBK * 2;              // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSmemAlloc = kStages * kStageBytes + 1024;
constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;

struct GemmBars {
  uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2], drain;
};

__global__ void __launch_bounds__(kThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tw,
                     __nv_bfloat16* __restrict__ c, int M, int N, int K, int32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ GemmBars bars;
  __shared__ uint32_t tmem_base;
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntn = (N + kBN - 1) / kBN;
  const int tiles = ((M + kBM - 1) / kBM) * ntn;
  const int nkb = (K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars.full[s]), 1);
      mbar_init(smem_u32(&bars.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars.acc_full[b]), 1);
      mbar_init(smem_u32(&bars.acc_empty[b]), kEpiWarps);
    }
    mbar_init(smem_u32(&bars.drain), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = tmem_base;
  auto fail = [&]() {
    atomicCAS(err, 0, PPS_DEV_ERR_WAIT_TIMEOUT);
    abort_flag = 1;
  };
  auto warp_wait = [&](uint64_t* bar, uint32_t parity, bool needed = true) {
    const bool ok = (!needed || mbar_wait(smem_u32(bar), parity)) && !abort_flag;
    return __all_sync(0xffffffffu, ok);
  };

  if (warp == 0) {
    // ------------------------------------------------------------- TMA producer
    if (lane == 0) {
      prefetch_tmap(&ta);
      prefetch_tmap(&tw);
    }
    int it = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
      const int m0 = (t / ntn) * kBM, n0 = (t % ntn) * kBN;
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const int s = it % kStages, use = it / kStages;
        if (!warp_wait(&bars.empty[s], (use - 1) & 1, use > 0)) { fail(); ok = false; break; }
        if (lane == 0) {
          const uint32_t fb = smem_u32(&bars.full[s]);
          const uint32_t base = smem_u32(smem + s * kStageBytes);
          mbar_expect_tx(fb, kStageBytes);
          tma_load_2d(base, &ta, kb * kBK, m0, fb);
          tma_load_2d(base + kABytes, &tw, kb * kBK, n0, fb);
        }
        __syncwarp();
      }
    }
    // every load started lands before the CTA may exit
    if (lane == 0) {
      const uint64_t lim = ok ? 2000000000ull : 10000000ull;
      for (int j = (it > kStages ? it - kStages : 0); j < it; ++j)
        mbar_wait(smem_u32(&bars.full[j % kStages]), (j / kStages) & 1, lim);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = idesc_bf16(kBM, kBN, 0, 0);
    int it = 0, tc = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x, ++tc) {
      const int b = tc & 1, use_b = tc >> 1;
      if (!warp_wait(&bars.acc_empty[b], (use_b - 1) & 1, use_b > 0)) { fail(); ok = false; break; }
      tc_fence_after();
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const int s = it % kStages;
        if (!warp_wait(&bars.full[s], (it / kStages) & 1)) { fail(); ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t a0 = smem_u32(smem + s * kStageBytes), w0 = a0 + kABytes;
#pragma unroll
          for (int ks = 0; ks < kBK / 16; ++ks)
            umma_ss(tm + b * kBN, smem_desc(a0 + ks * 32, 16, 1024),
                    smem_desc(w0 + ks * 32, 16, 1024), idesc, (kb > 0 || ks > 0) ? 1u : 0u);
          umma_commit(smem_u32(&bars.empty[s]));        // stage free once these MMAs finish
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) umma_commit(smem_u32(&bars.acc_full[b]));
      __syncwarp();
    }
    if (lane == 0) {
      umma_commit(smem_u32(&bars.drain));
      if (!mbar_wait(smem_u32(&bars.drain), 0)) fail();
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- epilogue
    const int quarter = warp & 3;                       // TMEM lanes this warp may read
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int r = quarter * 32 + lane;                  // row within the tile
    int tc = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++tc) {
      const int b = tc & 1, use_b = tc >> 1;
      if (!warp_wait(&bars.acc_full[b], use_b & 1)) { fail(); break; }
      tc_fence_after();
      const int m = (t / ntn) * kBM + r, n0 = (t % ntn) * kBN;
#pragma unroll 1
      for (int c0 = 0; c0 < kBN; c0 += 32) {
        uint32_t rr[32];
        tmem_ld32(tm + b * kBN + lane_off + c0, rr);
        tmem_wait_ld();
        if (m < M) {
          __nv_bfloat16* dst = c + (size_t)m * N + n0 + c0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (n0 + c0 + 8 * j >= N) break;
            int4 v;
            v.x = (int)pack_bf16(__uint_as_float(rr[8 * j + 0]), __uint_as_float(rr[8 * j + 1]));
            v.y = (int)pack_bf16(__uint_as_float(rr[8 * j + 2]), __uint_as_float(rr[8 * j + 3]));
            v.z = (int)pack_bf16(__uint_as_float(rr[8 * j + 4]), __uint_as_float(rr[8 * j + 5]));
            v.w = (int)pack_bf16(__uint_as_float(rr[8 * j + 6]), __uint_as_float(rr[8 * j + 7]));
            *reinterpret_cast<int4*>(dst + 8 * j) = v;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars.acc_empty[b]));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tm, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)f;
  });
  return fn;
}

// Row-major [rows, K] bf16 matrix; box = 64 columns x box_rows rows, 128-byte
// swizzle (the UMMA K-major layout); out-of-range elements read as zero.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace pps {

int launch_gemm_bf16(const void* a, const void* w, void* c, int32_t M, int32_t N, int32_t K,
                     int32_t* err, void* stream) {
  if (M == 0) return cudaSuccess;
  CUtensorMap ma, mw;
  if (!make_map(&ma, a, M, K, kBM) || !make_map(&mw, w, N, K, kBN))
    return (int)cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  if (e != cudaSuccess) return (int)e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return (int)e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return (int)e;
  const int64_t tiles = (int64_t)((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
  const int64_t grid = std::min<int64_t>(tiles, sms);
  gemm_bf16_kernel<<<(unsigned)grid, kThreads, kSmemAlloc, (cudaStream_t)stream>>>(
      ma, mw, (__nv_bfloat16*)c, M, N, K, err);
  count_launch();
  return (int)cudaGetLastError();
}

}  // namespace pps
