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
// Persistent kernel on CTA pairs (clusters of two CTAs, one CTA per SM): a
// pair computes 256 x 256 output tiles p, p + pairs, ... with tcgen05 MMAs of
// M = 256 issued by the even CTA (.cta_group::2): each CTA stages its own 128
// rows of A and its own 128 rows of W per K block, and each CTA's TMEM holds
// its 128 rows of the accumulator.  Per 64 of K an SM thus writes 32 KB into
// shared memory and its tensor core reads 32 KB there, against 48 + 48 KB for
// a 128 x 256 tile on one SM.  A stage holds 128 of K: the MMA warp waits on a
// stage barrier once per 8 MMAs, since that wait, not the data, is what kept
// the tensor pipe idle with 64-deep stages.  192 threads per CTA:
//   warp 0     TMA producer: per 128-wide K block, this CTA's A rows (128 x 128)
//              and W rows (128 x 128), each as two 64-column boxes with
//              128-byte swizzle, into a 3-stage ring (64 KB a stage);
//              completion is signalled on the even CTA's barrier, which
//              expects both CTAs' bytes;
//   warp 1     (even CTA) MMA issuer: 8 x tcgen05.mma (M 256, N 256, K 16) per K
//              block into one of two TMEM accumulators (2 x 256 columns), so the
//              epilogue of one tile overlaps the MMAs of the next; its commits
//              free the stage and announce the accumulator in both CTAs;
//   warps 2-5  epilogue: TMEM -> registers -> bf16 -> a 32 x 32 staging box in
//              shared memory (64-byte swizzle, two per warp) -> TMA store, row
//              = TMEM lane; the store writes whole 64-byte row pieces and
//              leaves out rows >= M and columns >= N; both CTAs' epilogue warps
//              release the accumulator on the even CTA's barrier.
// Every mbarrier wait is bounded; on timeout the kernel records
// PPS_DEV_ERR_WAIT_TIMEOUT and stops issuing.  No thread returns early: all of
// both CTAs meet at the closing cluster barrier, after the MMAs have drained,
// before the TMEM is freed.
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

constexpr int kBM = 128;                          // A rows per CTA (256 per pair)
constexpr int kBN = 256;                          // C columns per pair tile
constexpr int kBNh = kBN / 2;                     // W rows per CTA
constexpr int kBK = 128, kStages = 3;             // K block: two 64-column boxes per operand
constexpr int kSub = kBK / 64;
constexpr int kSubA = kBM * 64 * 2, kSubB = kBNh * 64 * 2;   // 16 KB each
constexpr int kABytes = kSub * kSubA;             // 32 KB
constexpr int kBBytes = kSub * kSubB;             // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;    // per CTA
constexpr int kEpiBox = 32;                       // output box: 32 rows x 32 columns
constexpr int kEpiBoxBytes = kEpiBox * kEpiBox * 2;  // 2 KB
constexpr int kRingBytes = kStages * kStageBytes;
constexpr int kSmemAlloc = kRingBytes + 4 * 2 * kEpiBoxBytes + 1024;
constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr uint16_t kPairMask = 0x3;

struct GemmBars {
  uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2], drain;
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tw,
                     const __grid_constant__ CUtensorMap tc, int M, int N, int K, int32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ GemmBars bars;
  __shared__ uint32_t tmem_base;
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();          // 0: issues the MMAs
  const int pair = (int)(blockIdx.x >> 1), pairs = (int)(gridDim.x >> 1);
  const int ntn = (N + kBN - 1) / kBN;
  const int tiles = ((M + 2 * kBM - 1) / (2 * kBM)) * ntn;
  const int nkb = (K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars.full[s]), 1);
      mbar_init(smem_u32(&bars.empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars.acc_full[b]), 1);
      mbar_init(smem_u32(&bars.acc_empty[b]), 2 * kEpiWarps);
    }
    mbar_init(smem_u32(&bars.drain), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&tmem_base), 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();                                   // the peer's barriers are initialised
  tc_fence_after();
  const uint32_t tm = tmem_base;
  auto fail = [&]() {
    atomicCAS(err, 0, PPS_DEV_ERR_WAIT_TIMEOUT);
    abort_flag = 1;
  };
  auto warp_wait = [&](uint64_t* bar, uint32_t parity, bool needed = true) -> bool {
    if (__all_sync(0xffffffffu, !needed || mbar_try_wait(smem_u32(bar), parity))) return true;
    const bool ok = (!needed || mbar_wait(smem_u32(bar), parity)) && !abort_flag;
    return __all_sync(0xffffffffu, ok) != 0;
  };

  if (warp == 0) {
    // ------------------------------------------------------------- TMA producer
    if (lane == 0) {
      prefetch_tmap(&ta);
      prefetch_tmap(&tw);
    }
    int it = 0;
    bool ok = true;
    for (int t = pair; ok && t < tiles; t += pairs) {
      const int m0 = (t / ntn) * (2 * kBM) + (int)rank * kBM;
      const int n0 = (t % ntn) * kBN + (int)rank * kBNh;
      for (int kb = 0; kb < nkb; ++kb, ++it) {
        const int s = it % kStages, use = it / kStages;
        if (!warp_wait(&bars.empty[s], (use - 1) & 1, use > 0)) { fail(); ok = false; break; }
        if (elect_one()) {
          const uint32_t fb = mapa_shared(smem_u32(&bars.full[s]), 0);
          const uint32_t base = smem_u32(smem + s * kStageBytes);
          if (rank == 0) mbar_expect_tx(smem_u32(&bars.full[s]), 2 * kStageBytes);
#pragma unroll
          for (int h = 0; h < kSub; ++h) {
            tma_load_2d_pair(base + h * kSubA, &ta, kb * kBK + h * 64, m0, fb);
            tma_load_2d_pair(base + kABytes + h * kSubB, &tw, kb * kBK + h * 64, n0, fb);
          }
        }
        __syncwarp();
      }
    }
    // the even CTA sees every load of both CTAs land before the pair may exit
    // (the odd CTA's loads are counted on the even CTA's barriers)
    if (rank == 0 && lane == 0) {
      const uint64_t lim = ok ? 2000000000ull : 10000000ull;
      for (int j = (it > kStages ? it - kStages : 0); j < it; ++j)
        mbar_wait(smem_u32(&bars.full[j % kStages]), (j / kStages) & 1, lim);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (rank == 0) {
      constexpr uint32_t idesc = idesc_bf16(2 * kBM, kBN, 0, 0);
      int it = 0, tc = 0;
      bool ok = true;
      for (int t = pair; ok && t < tiles; t += pairs, ++tc) {
        const int b = tc & 1, use_b = tc >> 1;
        if (!warp_wait(&bars.acc_empty[b], (use_b - 1) & 1, use_b > 0)) { fail(); ok = false; break; }
        tc_fence_after();
        for (int kb = 0; kb < nkb; ++kb, ++it) {
          const int s = it % kStages;
          if (!warp_wait(&bars.full[s], (it / kStages) & 1)) { fail(); ok = false; break; }
          tc_fence_after();
          if (elect_one()) {
            const uint32_t a0 = smem_u32(smem + s * kStageBytes);
            const uint64_t ad = smem_desc(a0, 16, 1024), wd = smem_desc(a0 + kABytes, 16, 1024);
#pragma unroll
            for (int ks = 0; ks < kBK / 16; ++ks)
              umma_ss_pair(tm + b * kBN, ad + (uint64_t)(((ks / 4) * kSubA + (ks % 4) * 32) >> 4),
                           wd + (uint64_t)(((ks / 4) * kSubB + (ks % 4) * 32) >> 4), idesc,
                           (kb > 0 || ks > 0) ? 1u : 0u);
            // the stage is free in both CTAs once these MMAs finish
            umma_commit_pair_mc(smem_u32(&bars.empty[s]), kPairMask);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (elect_one()) umma_commit_pair_mc(smem_u32(&bars.acc_full[b]), kPairMask);
        __syncwarp();
      }
      if (elect_one()) {
        umma_commit_pair(smem_u32(&bars.drain));
        if (!mbar_wait(smem_u32(&bars.drain), 0)) fail();
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int quarter = warp & 3;                       // TMEM lanes this warp may read
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t empty0 = mapa_shared(smem_u32(&bars.acc_empty[0]), 0);
    const uint32_t empty1 = mapa_shared(smem_u32(&bars.acc_empty[1]), 0);
    // two staging boxes per warp; with the 64-byte swizzle, 16-byte piece j of
    // row r sits at r * 64 + ((j ^ (r / 2 % 4)) * 16), so the 32 lanes' stores
    // of one piece each fill four distinct bank lines
    const uint32_t stage0 = smem_u32(smem + kRingBytes) + (uint32_t)(quarter * 2 * kEpiBoxBytes);
    const uint32_t row_off = (uint32_t)lane * 64u;
    const uint32_t sw = ((uint32_t)lane >> 1) & 3u;
    if (lane == 0) prefetch_tmap(&tc);
    int tc_i = 0, box = 0;
    for (int t = pair; t < tiles; t += pairs, ++tc_i) {
      const int b = tc_i & 1, use_b = tc_i >> 1;
      if (!warp_wait(&bars.acc_full[b], use_b & 1)) { fail(); break; }
      tc_fence_after();
      const int m_box = (t / ntn) * (2 * kBM) + (int)rank * kBM + quarter * 32;
      const int n0 = (t % ntn) * kBN;
#pragma unroll 1
      for (int c0 = 0; c0 < kBN; c0 += 32, ++box) {
        uint32_t rr[32];
        tmem_ld32(tm + b * kBN + lane_off + c0, rr);
        const uint32_t buf = stage0 + (uint32_t)(box & 1) * kEpiBoxBytes;
        if (box >= 2) {
          // the store issued from this box two rounds ago has read it
          if (lane == 0) bulk_wait_group_read<1>();
          __syncwarp();
        }
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t x = pack_bf16(__uint_as_float(rr[8 * j + 0]), __uint_as_float(rr[8 * j + 1]));
          const uint32_t y = pack_bf16(__uint_as_float(rr[8 * j + 2]), __uint_as_float(rr[8 * j + 3]));
          const uint32_t z = pack_bf16(__uint_as_float(rr[8 * j + 4]), __uint_as_float(rr[8 * j + 5]));
          const uint32_t w = pack_bf16(__uint_as_float(rr[8 * j + 6]), __uint_as_float(rr[8 * j + 7]));
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                           buf + row_off + ((((uint32_t)j) ^ sw) << 4)),
                       "r"(x), "r"(y), "r"(z), "r"(w)
                       : "memory");
        }
        fence_proxy_async_smem();                       // visible to the TMA store
        __syncwarp();
        if (lane == 0) {
          if (m_box < M && n0 + c0 < N) tma_store_2d(&tc, n0 + c0, m_box, buf);
          bulk_commit_group();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(b ? empty1 : empty0);
    }
    // the stores have read their boxes and written C before the CTA exits
    if (lane == 0) bulk_wait_group_all();
    __syncwarp();
  }

  // All MMAs of the pair have completed (the even CTA's drain), so both CTAs'
  // shared memory and TMEM may go.
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tm, 512);
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

// Row-major [rows, cols] bf16 matrix; box = box_cols x box_rows, the given
// swizzle (128-byte: the UMMA K-major layout of the operands); out-of-range
// elements read as zero and are not written.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows,
              int box_cols = 64, CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace pps {

int launch_gemm_bf16(const void* a, const void* w, void* c, int32_t M, int32_t N, int32_t K,
                     int32_t* err, void* stream) {
  if (M == 0) return cudaSuccess;
  CUtensorMap ma, mw, mc;
  if (!make_map(&ma, a, M, K, kBM) || !make_map(&mw, w, N, K, kBNh) ||
      !make_map(&mc, c, M, N, kEpiBox, kEpiBox, CU_TENSOR_MAP_SWIZZLE_64B))
    return (int)cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
  if (e != cudaSuccess) return (int)e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return (int)e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return (int)e;
  const int64_t tiles = (int64_t)((M + 2 * kBM - 1) / (2 * kBM)) * ((N + kBN - 1) / kBN);
  const int64_t grid = 2 * std::min<int64_t>(tiles, sms / 2);     // CTA pairs
  gemm_bf16_kernel<<<(unsigned)grid, kThreads, kSmemAlloc, (cudaStream_t)stream>>>(
      ma, mw, mc, M, N, K, err);
  count_launch();
  return (int)cudaGetLastError();
}

}  // namespace pps
