// Tensor-core attention tiles (tcgen05 + TMEM + TMA) for tasks with many query
// rows: prefill chunks, speculative-verify rows and wide shared-prefix groups.
//
// The matmul-softmax-matmul tile of the XY-Serve review ("Core claim"; Fig. 10
// pipeline of meta-attention) re-designed for sm_103a.  One CTA runs one task:
// 128 query rows (128 / G tokens x the G query heads of one kv head, so every
// K/V tile feeds all G heads) against the task's KV range in tiles of 128
// positions.  Fully masked causal tiles never reach the kernel (the planner
// stops each tile's KV range at its last token's causal limit; Fig. 11
// mask-aware computation).
//
// Warp roles (192 threads):
//   warps 0-3  softmax: thread m owns query row m = TMEM lane m.  Loads Q into
//              shared memory, turns S into P (online softmax in log2 units,
//              fp32), rescales O in TMEM when its reference max moves up by
//              more than 2^8, and writes the output or the partial (o, lse).
//   warp 4     TMA producer: K and V tiles, one 64-column box per page and
//              half of head_dim, into a 2-stage ring (128-byte swizzle).
//   warp 5     MMA issuer: S = Q K^T into one of two TMEM buffers, then
//              O += P V (P from shared memory, V MN-major), commits to mbarriers.
// Every mbarrier wait is bounded; on timeout the kernel records
// PPS_DEV_ERR_WAIT_TIMEOUT, stops issuing work and still frees TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "pps_internal.h"
#include "sm100_ptx.cuh"

namespace {

using namespace sm100;

constexpr int kThreads = 192;
constexpr int kStages = 2;
constexpr int kTile = 128;                    // KV positions per tile = query rows per task
constexpr float kRescaleThreshold = 8.f;      // log2 units

struct MmaParams {
  const pps::Task* tasks;
  const int32_t* rows;
  const int32_t* pages;
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  float* o_part;
  float* lse_part;
  int32_t* err;
  int32_t num_q_heads;
  int32_t G;
  int32_t page_size;
  float qk_scale;                             // sm_scale * log2(e)
};

struct Bars {
  uint64_t k_full[kStages], k_empty[kStages], v_full[kStages], v_empty[kStages];
  uint64_t s_full[2], s_free[2], p_full, o_done, q_full, drain;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
struct Layout {
  static constexpr int KB = D / 64;                  // 64-column blocks of head_dim
  static constexpr int kTileBytes = KB * 16384;      // 128 rows x D bf16
  static constexpr int q_off = 0;
  static constexpr int k_off = q_off + kTileBytes;
  static constexpr int v_off = k_off + kStages * kTileBytes;
  static constexpr int p_off = v_off + kStages * kTileBytes;
  static constexpr int bytes = p_off + 2 * 16384;    // P: 128 rows x 128 positions bf16
  static constexpr int smem_alloc = bytes + 1024;    // slack for 1024-byte alignment
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    mma_attention_kernel(const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv, const MmaParams p) {
  using Lay = Layout<D>;
  constexpr int KB = Lay::KB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ Bars bars;
  __shared__ uint32_t tmem_base;
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const pps::Task task = p.tasks[blockIdx.x];
  const int G = p.G;
  const int n_rows = task.n_tok * G;
  const int n_tiles = (task.kv_end - task.kv_begin + kTile - 1) / kTile;
  const uint32_t q_base = smem_u32(smem + Lay::q_off);
  const uint32_t k_base = smem_u32(smem + Lay::k_off);
  const uint32_t v_base = smem_u32(smem + Lay::v_off);
  const uint32_t p_base = smem_u32(smem + Lay::p_off);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars.k_full[s]), 1);
      mbar_init(smem_u32(&bars.k_empty[s]), 1);
      mbar_init(smem_u32(&bars.v_full[s]), 1);
      mbar_init(smem_u32(&bars.v_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&bars.s_full[b]), 1);
      mbar_init(smem_u32(&bars.s_free[b]), 4);
    }
    mbar_init(smem_u32(&bars.p_full), 4);
    mbar_init(smem_u32(&bars.o_done), 1);
    mbar_init(smem_u32(&bars.q_full), 4);
    mbar_init(smem_u32(&bars.drain), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(&tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = tmem_base;
  const uint32_t tm_s[2] = {tm, tm + 128};
  const uint32_t tm_o = tm + 256;

  auto fail = [&]() {
    atomicCAS(p.err, 0, PPS_DEV_ERR_WAIT_TIMEOUT);
    abort_flag = 1;
  };
  // A wait whose outcome is the same for every lane of the warp (the warp then
  // either goes on to warp-collective tcgen05 ld/st together or leaves together).
  auto warp_wait = [&](uint64_t* bar, uint32_t parity, bool needed = true) {
    const bool ok = (!needed || mbar_wait(smem_u32(bar), parity)) && !abort_flag;
    return __all_sync(0xffffffffu, ok);
  };

  if (warp < 4) {
    // ------------------------------------------------------------- softmax warps
    const int m = tid;                               // query row = TMEM lane
    const int i = m / G, g = m - (m / G) * G;
    const bool real = m < n_rows;
    const int h = task.kv_head * G + g;
    const int tok = real ? p.rows[task.row_off + i] : 0;
    // Q row -> swizzled shared memory (zeros for padding rows)
    {
      const int4* src = reinterpret_cast<const int4*>(p.q + ((size_t)tok * p.num_q_heads + h) * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const int4 v = real ? __ldg(src + c) : make_int4(0, 0, 0, 0);
        *reinterpret_cast<int4*>(smem + Lay::q_off + (c / 8) * 16384 + sw128(m, c % 8)) = v;
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bars.q_full));

    const int lim = real ? task.causal + i : -1;     // last visible position (inclusive)
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    float m_ref = -INFINITY, l_sum = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int b = j & 1;
      const int t0 = task.kv_begin + j * kTile;
      if (!warp_wait(&bars.s_full[b], (j >> 1) & 1)) { fail(); ok = false; break; }
      tc_fence_after();
      float s[kTile];
#pragma unroll
      for (int c0 = 0; c0 < kTile; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tm_s[b] + lane_off + c0, r);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) s[c0 + c] = __uint_as_float(r[c]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars.s_free[b]));

      const int bound = min(task.kv_end - t0, lim - t0 + 1);   // columns c < bound are visible
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < kTile; ++c) {
        s[c] = (c < bound) ? s[c] * p.qk_scale : -INFINITY;
        mx = fmaxf(mx, s[c]);
      }
      float m_use = m_ref, alpha = 1.f;
      if (mx > m_ref + kRescaleThreshold || m_ref == -INFINITY) {
        m_use = fmaxf(mx, m_ref);
        alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_use);
      }
      const float m_sub = (m_use == -INFINITY) ? 0.f : m_use;
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < kTile; ++c) {
        s[c] = ex2(s[c] - m_sub);                    // exp2(-inf) = 0 for masked columns
        rs += s[c];
      }
      l_sum = l_sum * alpha + rs;
      m_ref = m_use;
      // PV of the previous tile must be done before P and O are touched.
      if (j > 0) {
        if (!warp_wait(&bars.o_done, (j - 1) & 1)) { fail(); ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t r[32];
            tmem_ld32(tm_o + lane_off + c0, r);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
            tmem_st32(tm_o + lane_off + c0, r);
          }
          tmem_wait_st();
        }
      }
      // P row (bf16) -> swizzled shared memory, K-major over the tile's positions
#pragma unroll
      for (int c = 0; c < kTile / 8; ++c) {
        int4 v;
        v.x = (int)pack_bf16(s[8 * c + 0], s[8 * c + 1]);
        v.y = (int)pack_bf16(s[8 * c + 2], s[8 * c + 3]);
        v.z = (int)pack_bf16(s[8 * c + 4], s[8 * c + 5]);
        v.w = (int)pack_bf16(s[8 * c + 6], s[8 * c + 7]);
        *reinterpret_cast<int4*>(smem + Lay::p_off + (c / 8) * 16384 + sw128(m, c % 8)) = v;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars.p_full));
    }
    // epilogue: O / l
    if (ok && n_tiles > 0) {
      if (!warp_wait(&bars.o_done, (n_tiles - 1) & 1)) {
        fail();
      } else {
        tc_fence_after();
        const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
        const bool direct = task.out_pid < 0;
        const size_t prow = direct ? 0 : (size_t)(task.out_pid + i) * p.num_q_heads + h;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tm_o + lane_off + c0, r);
          tmem_wait_ld();
          if (real) {
            if (direct) {
              __nv_bfloat16* dst = p.out + ((size_t)tok * p.num_q_heads + h) * D + c0;
#pragma unroll
              for (int c = 0; c < 32; c += 8) {
                int4 v;
                v.x = (int)pack_bf16(__uint_as_float(r[c + 0]) * inv, __uint_as_float(r[c + 1]) * inv);
                v.y = (int)pack_bf16(__uint_as_float(r[c + 2]) * inv, __uint_as_float(r[c + 3]) * inv);
                v.z = (int)pack_bf16(__uint_as_float(r[c + 4]) * inv, __uint_as_float(r[c + 5]) * inv);
                v.w = (int)pack_bf16(__uint_as_float(r[c + 6]) * inv, __uint_as_float(r[c + 7]) * inv);
                *reinterpret_cast<int4*>(dst + c) = v;
              }
            } else {
              float* dst = p.o_part + prow * D + c0;
#pragma unroll
              for (int c = 0; c < 32; c += 4)
                *reinterpret_cast<float4*>(dst + c) =
                    make_float4(__uint_as_float(r[c]) * inv, __uint_as_float(r[c + 1]) * inv,
                                __uint_as_float(r[c + 2]) * inv, __uint_as_float(r[c + 3]) * inv);
            }
          }
        }
        if (real && !direct)
          p.lse_part[prow] = l_sum > 0.f ? m_ref + __log2f(l_sum) : -INFINITY;
      }
    }
  } else if (warp == 4) {
    // ------------------------------------------------------------- TMA producer
    // Lane 0 arms each stage's barrier with the tile's byte count, then one
    // lane per (page, 64-column block) issues its box: a single issuing thread
    // cannot issue small TMA loads fast enough to keep the tensor core fed.
    if (lane == 0) {
      prefetch_tmap(&tmk);
      prefetch_tmap(&tmv);
    }
    const int P = p.page_size;
    const uint32_t box_bytes = (uint32_t)P * 128u;
    int issued = 0;
    bool ok = true;
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int st = j % kStages, use = j / kStages;
      const int t0 = task.kv_begin + j * kTile;
      const int valid = min(kTile, task.kv_end - t0);
      const int npg = (valid + P - 1) / P;
      const uint32_t bytes = (uint32_t)(npg * KB) * box_bytes;
      const int pg = lane / KB, kb = lane % KB;
      const bool mine = lane < npg * KB;
      const int page = mine ? p.pages[task.page_off + (t0 + pg * P) / P] : 0;
      const uint32_t kf = smem_u32(&bars.k_full[st]);
      if (!warp_wait(&bars.k_empty[st], (use - 1) & 1, use > 0)) { fail(); ok = false; break; }
      if (lane == 0) mbar_expect_tx(kf, bytes);
      __syncwarp();
      if (mine)
        tma_load_4d(k_base + st * Lay::kTileBytes + kb * 16384 + pg * P * 128, &tmk, kb * 64, 0,
                    task.kv_head, page, kf);
      const uint32_t vf = smem_u32(&bars.v_full[st]);
      if (!warp_wait(&bars.v_empty[st], (use - 1) & 1, use > 0)) { fail(); ok = false; break; }
      if (lane == 0) mbar_expect_tx(vf, bytes);
      __syncwarp();
      if (mine)
        tma_load_4d(v_base + st * Lay::kTileBytes + kb * 16384 + pg * P * 128, &tmv, kb * 64, 0,
                    task.kv_head, page, vf);
      issued = j + 1;
    }
    // Before the CTA can exit, every load it started must have landed.
    if (lane == 0) {
      for (int j = (issued > kStages ? issued - kStages : 0); j < issued; ++j) {
        const int st = j % kStages, use = j / kStages;
        mbar_wait(smem_u32(&bars.k_full[st]), use & 1, ok ? 2000000000ull : 10000000ull);
        mbar_wait(smem_u32(&bars.v_full[st]), use & 1, ok ? 2000000000ull : 10000000ull);
      }
    }
  } else {
    // ------------------------------------------------------------- MMA issuer
    constexpr uint32_t id_qk = idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t id_pv = idesc_bf16(128, D, 0, 1);
    bool ok = warp_wait(&bars.q_full, 0);
    if (!ok) fail();
    for (int j = 0; ok && j <= n_tiles; ++j) {
      if (j < n_tiles) {
        const int st = j % kStages, b = j & 1;
        if (!warp_wait(&bars.k_full[st], (j / kStages) & 1)) { fail(); break; }
        if (j >= 2 && !warp_wait(&bars.s_free[b], ((j - 2) >> 1) & 1)) { fail(); break; }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t kt = k_base + st * Lay::kTileBytes;
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = (ks / 4) * 16384 + (ks % 4) * 32;
            umma_ss(tm_s[b], smem_desc(q_base + off, 16, 1024), smem_desc(kt + off, 16, 1024),
                    id_qk, ks > 0);
          }
          umma_commit(smem_u32(&bars.s_full[b]));
          umma_commit(smem_u32(&bars.k_empty[st]));
        }
        __syncwarp();
      }
      if (j >= 1) {
        const int jj = j - 1, st = jj % kStages;
        if (!warp_wait(&bars.p_full, jj & 1)) { fail(); break; }
        if (!warp_wait(&bars.v_full[st], (jj / kStages) & 1)) { fail(); break; }
        const int valid = min(kTile, task.kv_end - (task.kv_begin + jj * kTile));
        if (valid < kTile) {
          // Rows past the task's last position may hold anything (NaN included);
          // P is 0 there, and 0 * NaN would poison O, so clear them.
          uint8_t* vt = smem + Lay::v_off + st * Lay::kTileBytes;
          for (int idx = lane; idx < (kTile - valid) * 8 * KB; idx += 32) {
            const int kb = idx / ((kTile - valid) * 8);
            const int rem = idx - kb * (kTile - valid) * 8;
            const int r = valid + rem / 8, c = rem % 8;
            *reinterpret_cast<int4*>(vt + kb * 16384 + r * 128 + c * 16) = make_int4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t vt = v_base + st * Lay::kTileBytes;
#pragma unroll
          for (int ks = 0; ks < kTile / 16; ++ks) {
            const uint32_t aoff = (ks / 4) * 16384 + (ks % 4) * 32;
            umma_ss(tm_o, smem_desc(p_base + aoff, 16, 1024), smem_desc(vt + ks * 2048, 16384, 1024),
                    id_pv, (jj > 0 || ks > 0) ? 1u : 0u);
          }
          umma_commit(smem_u32(&bars.o_done));
          umma_commit(smem_u32(&bars.v_empty[st]));
        }
        __syncwarp();
      }
    }
    // Every MMA this warp issued has completed before TMEM is freed.
    if (lane == 0) {
      umma_commit(smem_u32(&bars.drain));
      if (!mbar_wait(smem_u32(&bars.drain), 0)) fail();
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tm, 512);
  }
}

// ---- host: tensor maps over the pool ------------------------------------------------

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

// 4-D view [num_pages][Hkv][P][D] of one pool array; box = 64 columns x P slots
// of one page and kv head, 128-byte swizzle (matches the UMMA K-major layout).
bool make_pool_map(CUtensorMap* map, const void* base, const pps_pool& pool) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int D = pool.head_dim, P = pool.page_size, H = pool.num_kv_heads;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)P, (cuuint64_t)H, (cuuint64_t)pool.num_pages};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)P * D * 2, (cuuint64_t)H * P * D * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)P, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
int launch_t(const pps::Shape& s, const pps::DeviceTables& t, int64_t n, const void* q,
             const pps_pool& pool, void* out, int32_t* err, cudaStream_t st) {
  CUtensorMap mk, mv;
  if (!make_pool_map(&mk, pool.k, pool) || !make_pool_map(&mv, pool.v, pool))
    return (int)cudaErrorInvalidValue;
  auto kern = mma_attention_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Layout<D>::smem_alloc);
  if (e != cudaSuccess) return (int)e;
  MmaParams prm{t.mma_tasks, t.rows, t.pages, (const __nv_bfloat16*)q, (__nv_bfloat16*)out,
                t.o_part, t.lse_part, err, s.num_q_heads, s.group, s.page_size,
                s.sm_scale * 1.4426950408889634f};
  kern<<<(unsigned)n, kThreads, Layout<D>::smem_alloc, st>>>(mk, mv, prm);
  pps::count_launch();
  return (int)cudaGetLastError();
}

}  // namespace

namespace pps {

bool mma_path_available() { return true; }

int launch_mma_attention(const Shape& s, const DeviceTables& t, int64_t num_tasks, const void* q,
                         const pps_pool& pool, void* out, int32_t* err, void* stream) {
  if (num_tasks == 0) return cudaSuccess;
  auto st = (cudaStream_t)stream;
  if (s.head_dim == 128) return launch_t<128>(s, t, num_tasks, q, pool, out, err, st);
  return launch_t<64>(s, t, num_tasks, q, pool, out, err, st);
}

}  // namespace pps
