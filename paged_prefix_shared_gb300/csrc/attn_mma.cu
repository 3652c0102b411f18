// Tensor-core attention tiles (tcgen05 + TMEM + TMA) for tasks with many query
// rows: prefill chunks, speculative-verify rows and wide shared-prefix groups.
//
// The matmul-softmax-matmul tile of the XY-Serve review ("Core claim"; Fig. 10,
// pipeline of meta-attention, where the cube works on one tile while the
// vector unit runs the softmax of another) re-designed for sm_103a.
//
// A task holds up to 256 query rows of one kv head: two 128-row tiles A and B
// (row = token * G + head, so every K/V tile feeds all G heads) that share the
// task's KV range.  The tensor core alternates between them: while softmax
// warpgroup A turns S_A into P_A, the MMA warp runs PV_B and QK_B on tile B,
// and the other way round.  Each tile skips the KV tiles past its own causal
// limit, and fully masked tiles never exist (the planner stops each task's
// range at its last token's limit; Fig. 11, mask-aware computation).  Draft-
// tree rows (Fig. 8, tree-based speculation) also mask the draft positions
// that are not their ancestors, in the KV tiles their 64-key window reaches.
//
// Warp roles (352 threads, one persistent CTA per SM taking tasks in
// symmetric round-robin order over the work-sorted list):
//   warps 0-3  softmax A, warps 4-7 softmax B: thread m of a warpgroup owns
//              query row m = TMEM lane m.  It loads its Q row into 128-byte
//              swizzled shared memory, turns its S row into P in one pass over
//              TMEM against its running reference max (two passes, and an O
//              rescale in TMEM, only when a score exceeds that reference by more
//              than 2^8), writes P as bf16 over S's own columns, and writes the
//              output row or the partial (o, lse).
//   warps 8/10 TMA producers of K and of V: tiles of 128 positions (one box
//              per page and 64-column block, issued by one lane each) into a
//              2-stage ring each.  Two warps, so that a K tile whose stage has
//              freed never queues behind the V tile's issue (with 16-position
//              pages a tile is 16 boxes).
//   warp 9     MMA issuer: S_X = Q_X K^T (both K-major in shared memory) and
//              O_X += P_X V (P from TMEM, V MN-major in shared memory), in the
//              order PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1).
// TMEM (512 columns): S_A | S_B | O_A | O_B.  Every mbarrier wait is bounded;
// on timeout the kernel records PPS_DEV_ERR_WAIT_TIMEOUT, stops issuing work,
// drains what it issued and still frees TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <type_traits>
#include <mutex>

#include "pps_internal.h"
#include "sm100_ptx.cuh"
#include "append_dev.cuh"

namespace {

using namespace sm100;

constexpr int kSoftmaxWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kProducerVWarp = 10;
constexpr int kThreads = 352;
constexpr int kStages = 2;
constexpr int kTile = 128;                    // KV positions per tile = query rows per tile
constexpr float kRescaleThreshold = 8.f;      // log2 units
constexpr float kRescaleSum = 256.f;          // 2^kRescaleThreshold

struct MmaParams {
  const pps::Task* tasks;
  int32_t num_tasks;
  const int32_t* rows;
  const int32_t* pages;
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  float* o_part;
  float* lse_part;
  int32_t* err;
  const unsigned long long* tree_mask;        // per token lookback masks, or nullptr
  int32_t num_q_heads;
  int32_t G;
  int32_t page_size;
  float qk_scale;                             // sm_scale * log2(e)
  // the step's rows to append first (num_tokens 0: none), into the pool
  pps::AppendArgs append;
  void* pool_k;
  void* pool_v;
  int32_t num_kv_heads;
  int32_t num_pages;
  int32_t* sync;
};

struct Bars {
  uint64_t k_full[kStages], k_empty[kStages], v_full[kStages], v_empty[kStages];
  uint64_t s_full[2], p_full[2], o_done[2], q_full, drain;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ int snake_task(int ti, int b, int C) {
  return ti * C + ((ti & 1) ? (C - 1 - b) : b);
}

// OR of `pred` over the 256 softmax threads (named barrier 1); every softmax
// thread gets the same answer.
__device__ __forceinline__ bool softmax_barrier_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n"
      " bar.red.or.pred po, 1, 256, pi;\n selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

// Bit c of the result is bit c + s of `rev` where 0 <= c + s < 64, else 1.
__device__ __forceinline__ unsigned long long window64(unsigned long long rev, int s) {
  if (s >= 64 || s <= -64) return ~0ull;
  if (s >= 0) return (rev >> s) | (s ? (~0ull << (64 - s)) : 0ull);
  return (rev << -s) | ((1ull << -s) - 1ull);
}

// Columns [0, n) of a 64-column word.
__device__ __forceinline__ unsigned long long low_bits(int n) {
  return n >= 64 ? ~0ull : (n <= 0 ? 0ull : ((1ull << n) - 1ull));
}

template <int D>
struct Layout {
  static constexpr int KB = D / 64;                  // 64-column blocks of head_dim
  static constexpr int kTileBytes = KB * 16384;      // 128 rows x D bf16
  static constexpr int q_off = 0;                    // Q_A, Q_B
  static constexpr int k_off = q_off + 2 * kTileBytes;
  static constexpr int v_off = k_off + kStages * kTileBytes;
  static constexpr int bytes = v_off + kStages * kTileBytes;
  static constexpr int smem_alloc = bytes + 1024;    // slack for 1024-byte alignment
};

// Per task and tile X: real rows and the number of 128-position KV tiles the
// tile attends to (its last token's causal limit may end before the task's).
struct TileRange {
  int rows;
  int n_tiles;
};
__device__ __forceinline__ TileRange tile_range(const pps::Task& t, int X, int G) {
  const int n_rows = t.n_tok * G;
  TileRange r;
  r.rows = min(max(n_rows - X * 128, 0), 128);
  if (r.rows == 0) {
    r.n_tiles = 0;
    return r;
  }
  const int last_tok = (X * 128 + r.rows - 1) / G;
  int end = t.kv_end;
  if (t.causal != PPS_NO_CAUSAL) end = min(end, t.causal + last_tok + 1);
  r.n_tiles = (end - t.kv_begin + kTile - 1) / kTile;
  return r;
}

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
  // The CTA's next task, read during the current one (see the softmax warps):
  // its record per tile, and per softmax thread its token (-1: padding row),
  // query head and draft-tree lookback mask.
  __shared__ pps::Task next_task[2];
  __shared__ int2 next_row[kSoftmaxWarps * 32];
  __shared__ unsigned long long next_mask[kSoftmaxWarps * 32];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x, nctas = gridDim.x;
  const int G = p.G;
  const uint32_t q_base = smem_u32(smem + Lay::q_off);
  const uint32_t k_base = smem_u32(smem + Lay::k_off);
  const uint32_t v_base = smem_u32(smem + Lay::v_off);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars.k_full[s]), 1);
      mbar_init(smem_u32(&bars.k_empty[s]), 1);
      mbar_init(smem_u32(&bars.v_full[s]), 1);
      mbar_init(smem_u32(&bars.v_empty[s]), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&bars.s_full[x]), 1);
      mbar_init(smem_u32(&bars.p_full[x]), 4);
      mbar_init(smem_u32(&bars.o_done[x]), 1);
    }
    mbar_init(smem_u32(&bars.q_full), kSoftmaxWarps);
    mbar_init(smem_u32(&bars.drain), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = tmem_base;
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
  // A wait whose outcome is the same for every lane of the warp (the warp then
  // goes on to warp-collective tcgen05 ld/st together, or leaves together).
  // The abort flag is read only when the phase has not completed at the first
  // poll (a shared-memory load in every wait slowed the MMA issuer).
  auto warp_wait = [&](uint64_t* bar, uint32_t parity, bool needed = true) -> bool {
    if (__all_sync(0xffffffffu, !needed || mbar_try_wait(smem_u32(bar), parity))) return true;
    const bool ok = (!needed || mbar_wait(smem_u32(bar), parity)) && !abort_flag;
    return __all_sync(0xffffffffu, ok) != 0;
  };

  if (warp < kSoftmaxWarps) {
    // ------------------------------------------------------------- softmax warps
    const int X = warp >> 2;                        // tile of this warpgroup
    const int m = tid & 127;                        // row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tm_s = tm + X * 128;             // S_X, and P_X over its first 64 columns
    const uint32_t tm_o = tm + 256 + X * D;         // O_X
    uint8_t* q_tile = smem + Lay::q_off + X * Lay::kTileBytes;
    int sx = 0, ox = 0;                             // phases consumed on s_full[X] / o_done[X]
    // A task switch costs a CTA ~10 us of mostly idle tensor core (epilogue,
    // Q rows, first S): the chain of dependent loads task -> token -> Q row
    // alone took ~3 us.  So during a task, after its first tile, each thread
    // reads the next task's record, its token and mask into shared memory
    // (`meta`), and once this tile's last QK has completed (the last s_full)
    // it starts the copy of its next Q row into the now free Q tile (`q_pref`).
    bool meta = false, q_pref = false;
    for (int ti = 0;; ++ti) {
      const int t = snake_task(ti, b, nctas);
      // Both warpgroups start a task together (and stop together): neither can
      // run a task ahead and complete the next task's q_full phase alone.
      if (softmax_barrier_or(t >= p.num_tasks || abort_flag)) break;
      const pps::Task task = meta ? next_task[X] : p.tasks[t];
      const TileRange tr = tile_range(task, X, G);
      const int r = X * 128 + m;                    // row within the task
      const bool real = m < tr.rows;
      const int i = r / G, g = r - (r / G) * G;
      const int h = task.kv_head * G + g;
      const int tok = meta ? max(next_row[tid].x, 0) : (real ? p.rows[task.row_off + i] : 0);
      const unsigned long long tmask_pre = meta ? next_mask[tid] : ~0ull;
      // Q row -> swizzled shared memory (zeros for padding rows).  Every MMA of
      // the previous task completed before its epilogues, which precede this.
      if (q_pref) {
        cp_async_wait_all();
      } else {
        const int4* src = reinterpret_cast<const int4*>(p.q + ((size_t)tok * p.num_q_heads + h) * D);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const int4 v = real ? __ldg(src + c) : make_int4(0, 0, 0, 0);
          *reinterpret_cast<int4*>(q_tile + (c / 8) * 16384 + sw128(m, c % 8)) = v;
        }
      }
      const bool had_meta = meta;
      meta = q_pref = false;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars.q_full));
      if (tr.n_tiles == 0) continue;

      const int lim = real ? task.causal + i : -1;  // last visible position (inclusive)
      // Draft-tree rows: bit k of the lookback mask = the key k positions
      // before the row's own one is visible.  Kept bit-reversed so the
      // visibility of a tile's columns is a shifted window of it.
      const unsigned long long tmask =
          had_meta ? tmask_pre
                   : ((p.tree_mask && real && task.causal != PPS_NO_CAUSAL) ? p.tree_mask[tok] : ~0ull);
      const bool trow = tmask != ~0ull;
      const unsigned long long trev = __brevll(tmask);
      // Padding rows see no key: any finite reference keeps their P at 0 and
      // keeps them off the exact path below.
      float m_ref = real ? -INFINITY : 0.f, l_sum = 0.f;
      bool ok = true;
      for (int j = 0; j < tr.n_tiles; ++j, ++sx) {
        const int t0 = task.kv_begin + j * kTile;
        if (!warp_wait(&bars.s_full[X], sx & 1)) { fail(); ok = false; break; }
        if (meta && j + 1 == tr.n_tiles) {
          // this tile's last QK has completed: Q_X is free for the next task
          const int2 nr = next_row[tid];
          const char* src = reinterpret_cast<const char*>(
              p.q + ((size_t)max(nr.x, 0) * p.num_q_heads + nr.y) * D);
#pragma unroll
          for (int c = 0; c < D / 8; ++c)
            cp_async16(smem_u32(q_tile + (c / 8) * 16384 + sw128(m, c % 8)), src + c * 16,
                       nr.x >= 0 ? 16u : 0u);
          q_pref = true;
        }
        tc_fence_after();
        const int bound = min(task.kv_end - t0, lim - t0 + 1);     // columns c < bound visible
        // the row's tree window [lim - 63, lim] reaches into this tile
        const bool tree_here = trow && t0 + kTile - 1 >= lim - 63;
        const bool full = __all_sync(0xffffffffu, bound >= kTile && !tree_here);
        // Visible columns (when not full): bit c of vis[c / 64].
        unsigned long long vis[2] = {~0ull, ~0ull};
        if (!full) {
          vis[0] = low_bits(bound);
          vis[1] = low_bits(bound - 64);
          if (tree_here) {
            vis[0] &= window64(trev, 63 - (lim - t0));
            vis[1] &= window64(trev, 127 - (lim - t0));
          }
        }
        // Hot path (a tile with every column visible, after the row's first):
        // one pass against the running reference, P = exp2(s * scale - m_ref),
        // two columns per packed multiply-add, S read in two 64-column halves.
        // Valid unless a score exceeds the reference by the threshold, which
        // makes some P exceed 2^8 and so the row's sum.  Everything else
        // (masked tiles, first tiles, a reference that must move) takes the
        // exact two-pass path below, written as rolled loops.  The hot path is
        // one straight block of code and the rest stays out of its way: the
        // instruction cache is shared by every warp of a scheduler, and the MMA
        // issuer stalls whenever the softmax code pushes its instructions out.
        // A row's first tile with every column visible: its maximum becomes
        // the reference, and the tile takes the hot path.
        if (__all_sync(0xffffffffu, full && m_ref == -INFINITY)) {
          float mx = -INFINITY;
#pragma unroll 1
          for (int c0 = 0; c0 < kTile; c0 += 32) {
            uint32_t rr[32];
            tmem_ld32(tm_s + lane_off + c0, rr);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) mx = fmaxf(mx, __uint_as_float(rr[c]));
          }
          m_ref = mx * p.qk_scale;
        }
        // A masked tile after the row's first: -inf over the invisible
        // columns of S (chunks with every column visible are skipped), and
        // the tile takes the hot path like a full one.
        bool masked = false;
        if (!full && __all_sync(0xffffffffu, m_ref != -INFINITY)) {
#pragma unroll 1
          for (int c0 = 0; c0 < kTile; c0 += 32) {
            const uint32_t vb = (uint32_t)((c0 < 64 ? vis[0] : vis[1]) >> (c0 & 63));
            if (__any_sync(0xffffffffu, vb != ~0u)) {
              uint32_t rr[32];
              tmem_ld32(tm_s + lane_off + c0, rr);
              tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < 32; ++c)
                if (!((vb >> c) & 1u)) rr[c] = 0xff800000u;
              tmem_st32(tm_s + lane_off + c0, rr);
            }
          }
          tmem_wait_st();
          masked = true;
        }
        float rs0 = 0.f, rs1 = 0.f, alpha = 1.f, m_use = m_ref;
        bool exact = !__all_sync(0xffffffffu, (full || masked) && m_ref != -INFINITY);
        if (!exact) {
          const uint64_t sc2 = f32x2(p.qk_scale, p.qk_scale);
          const uint64_t nm2 = f32x2(-m_ref, -m_ref);
          uint32_t pk[kTile / 2];                  // P row, bf16 pairs, stored once verified
#pragma unroll
          for (int h = 0; h < kTile; h += 64) {
            uint32_t ra[32], rb[32];
            tmem_ld32(tm_s + lane_off + h, ra);
            tmem_ld32(tm_s + lane_off + h + 32, rb);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
              float a, bb;
              ffma2(a, bb, __uint_as_float(c < 32 ? ra[c] : rb[c - 32]),
                    __uint_as_float(c < 32 ? ra[c + 1] : rb[c - 31]), sc2, nm2);
              a = ex2(a);
              bb = ex2(bb);
              fadd2(rs0, rs1, a, bb);
              pk[(h + c) / 2] = pack_bf16(a, bb);
            }
          }
          exact = __any_sync(0xffffffffu, rs0 + rs1 > kRescaleSum);
          if (!exact) {
            // P over S's first 64 columns (S has been read in full above)
#pragma unroll
            for (int c0 = 0; c0 < kTile / 2; c0 += 16) {
              uint32_t w[16];
#pragma unroll
              for (int c = 0; c < 16; ++c) w[c] = pk[c0 + c];
              tmem_st16(tm_s + lane_off + c0, w);
            }
          }
        }
        if (exact) {
          // Pass 1: the row maximum of the visible scores (rolled: rare code).
          float mx = -INFINITY;
#pragma unroll 1
          for (int c0 = 0; c0 < kTile; c0 += 32) {
            uint32_t rr[32];
            tmem_ld32(tm_s + lane_off + c0, rr);
            tmem_wait_ld();
            const uint32_t vb =
                full ? ~0u : (uint32_t)((c0 < 64 ? vis[0] : vis[1]) >> (c0 & 63));
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if ((vb >> c) & 1u) mx = fmaxf(mx, __uint_as_float(rr[c]));
          }
          const float mxs = (mx == -INFINITY) ? -INFINITY : mx * p.qk_scale;
          if (mxs > m_ref + kRescaleThreshold || (m_ref == -INFINITY && mxs != -INFINITY)) {
            m_use = fmaxf(mxs, m_ref);
            alpha = (m_ref == -INFINITY) ? 0.f : ex2(m_ref - m_use);
          }
          // O rescale: the PV of this tile's previous KV tile completed before
          // this S was delivered (one in-order tcgen05 stream; the commit behind
          // s_full covers both).
          if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t ro[32];
              tmem_ld32(tm_o + lane_off + c0, ro);
              tmem_wait_ld();
#pragma unroll
              for (int c = 0; c < 32; ++c) ro[c] = __float_as_uint(__uint_as_float(ro[c]) * alpha);
              tmem_st32(tm_o + lane_off + c0, ro);
            }
          }
          // Pass 2: P = exp2(s * scale - m); chunk c0 is stored over columns
          // c0/2 .. c0/2 + 15, all of which this pass has already read.
          const float msub = (m_use == -INFINITY) ? 0.f : m_use;
          const uint64_t sc2 = f32x2(p.qk_scale, p.qk_scale);
          const uint64_t nm2 = f32x2(-msub, -msub);
          rs0 = rs1 = 0.f;
#pragma unroll 1
          for (int c0 = 0; c0 < kTile; c0 += 32) {
            uint32_t rr[32];
            tmem_ld32(tm_s + lane_off + c0, rr);
            tmem_wait_ld();
            const uint32_t vb =
                full ? ~0u : (uint32_t)((c0 < 64 ? vis[0] : vis[1]) >> (c0 & 63));
            uint32_t w[16];
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              const float sa = ((vb >> c) & 1u) ? __uint_as_float(rr[c]) : -INFINITY;
              const float sb = ((vb >> (c + 1)) & 1u) ? __uint_as_float(rr[c + 1]) : -INFINITY;
              float a, bb;
              ffma2(a, bb, sa, sb, sc2, nm2);
              a = ex2(a);
              bb = ex2(bb);
              fadd2(rs0, rs1, a, bb);
              w[c / 2] = pack_bf16(a, bb);
            }
            tmem_st16(tm_s + lane_off + c0 / 2, w);
          }
        }
        const float rs = rs0 + rs1;
        m_ref = m_use;
        l_sum = l_sum * alpha + rs;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars.p_full[X]));
        if (j == 0) {
          // the next task's record, token and mask, read while the tensor
          // core runs this tile's PV and the next QK
          const int tn = snake_task(ti + 1, b, nctas);
          if (tn < p.num_tasks) {
            const pps::Task nt = p.tasks[tn];
            const TileRange ntr = tile_range(nt, X, G);
            const bool nreal = m < ntr.rows;
            const int ni = r / G;
            const int ntok = nreal ? p.rows[nt.row_off + ni] : -1;
            next_row[tid] = make_int2(ntok, nt.kv_head * G + g);
            next_mask[tid] = (p.tree_mask && nreal && nt.causal != PPS_NO_CAUSAL)
                                 ? p.tree_mask[ntok] : ~0ull;
            if (m == 0) next_task[X] = nt;
            meta = true;
          }
        }
      }
      if (!ok) continue;                            // the next task barrier sees the abort
      // epilogue: O / l once the task's last PV on this tile is done
      if (!warp_wait(&bars.o_done[X], ox & 1)) {
        fail();
        continue;
      }
      ++ox;
      tc_fence_after();
      const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
      const bool direct = task.out_pid < 0;
      const size_t prow = direct ? 0 : (size_t)(task.out_pid + i) * p.num_q_heads + h;
      // With G a multiple of 4, the 4 lanes of each lane quad hold one token's
      // 4 consecutive heads, rows that are contiguous in the output: a 4 x 4
      // transpose of 16-byte pieces across the quad lets every store of the
      // warp write 64 contiguous bytes per quad instead of 16 scattered ones.
      const bool quads = direct && (G & 3) == 0;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t rr[32];
        tmem_ld32(tm_o + lane_off + c0, rr);
        tmem_wait_ld();
        if (quads) {
          int4 pc[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t* v = rr + 8 * q;
            pc[q].x = (int)pack_bf16(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv);
            pc[q].y = (int)pack_bf16(__uint_as_float(v[2]) * inv, __uint_as_float(v[3]) * inv);
            pc[q].z = (int)pack_bf16(__uint_as_float(v[4]) * inv, __uint_as_float(v[5]) * inv);
            pc[q].w = (int)pack_bf16(__uint_as_float(v[6]) * inv, __uint_as_float(v[7]) * inv);
          }
          const int k = lane & 3;
          auto xchg = [&](int4& a, int4& b, bool hi, int mask) {
            // send b (hi lanes send a), receive into the slot that was sent
            int4 s = hi ? a : b, r;
            r.x = __shfl_xor_sync(0xffffffffu, s.x, mask);
            r.y = __shfl_xor_sync(0xffffffffu, s.y, mask);
            r.z = __shfl_xor_sync(0xffffffffu, s.z, mask);
            r.w = __shfl_xor_sync(0xffffffffu, s.w, mask);
            if (hi) a = r; else b = r;
          };
          xchg(pc[0], pc[2], (k & 2) != 0, 2);
          xchg(pc[1], pc[3], (k & 2) != 0, 2);
          xchg(pc[0], pc[1], (k & 1) != 0, 1);
          xchg(pc[2], pc[3], (k & 1) != 0, 1);
          // lane k now holds piece k of the quad's rows 0..3
          if (real) {
            __nv_bfloat16* grp = p.out + ((size_t)tok * p.num_q_heads + (h - k)) * D + c0 + 8 * k;
#pragma unroll
            for (int q = 0; q < 4; ++q) *reinterpret_cast<int4*>(grp + (size_t)q * D) = pc[q];
          }
          continue;
        }
        if (real) {
          if (direct) {
            __nv_bfloat16* dst = p.out + ((size_t)tok * p.num_q_heads + h) * D + c0;
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
              int4 v;
              v.x = (int)pack_bf16(__uint_as_float(rr[c + 0]) * inv, __uint_as_float(rr[c + 1]) * inv);
              v.y = (int)pack_bf16(__uint_as_float(rr[c + 2]) * inv, __uint_as_float(rr[c + 3]) * inv);
              v.z = (int)pack_bf16(__uint_as_float(rr[c + 4]) * inv, __uint_as_float(rr[c + 5]) * inv);
              v.w = (int)pack_bf16(__uint_as_float(rr[c + 6]) * inv, __uint_as_float(rr[c + 7]) * inv);
              *reinterpret_cast<int4*>(dst + c) = v;
            }
          } else {
            float* dst = p.o_part + prow * D + c0;
#pragma unroll
            for (int c = 0; c < 32; c += 4)
              *reinterpret_cast<float4*>(dst + c) =
                  make_float4(__uint_as_float(rr[c]) * inv, __uint_as_float(rr[c + 1]) * inv,
                              __uint_as_float(rr[c + 2]) * inv, __uint_as_float(rr[c + 3]) * inv);
          }
        }
      }
      if (real && !direct) p.lse_part[prow] = l_sum > 0.f ? m_ref + __log2f(l_sum) : -INFINITY;
      tc_fence_before();       // the O reads finish before the next task's first PV
    }
    cp_async_wait_all();       // a prefetched row of a task that never started
  } else if (warp == kProducerWarp || warp == kProducerVWarp) {
    // ------------------------------------------------------------- TMA producers
    // (K in warp 8, V in warp 10.)  Lane 0 arms a stage's barrier with the
    // tile's byte count, then one lane per (page, 64-column block) issues its
    // box: a single issuing thread cannot issue small TMA loads fast enough to
    // keep the tensor core fed.
    const bool is_k = warp == kProducerWarp;
    const CUtensorMap* map = is_k ? &tmk : &tmv;
    const uint32_t ring = is_k ? k_base : v_base;
    uint64_t* full = is_k ? bars.k_full : bars.v_full;
    uint64_t* empty = is_k ? bars.k_empty : bars.v_empty;
    if (lane == 0) prefetch_tmap(map);
    const int P = p.page_size;
    const uint32_t box_bytes = (uint32_t)P * 128u;
    int it = 0;                                     // KV tiles loaded by this CTA
    bool ok = true;
    int t;
    for (int ti = 0; ok && (t = snake_task(ti, b, nctas)) < p.num_tasks; ++ti) {
      const pps::Task task = p.tasks[t];
      const int n_tiles = max(tile_range(task, 0, G).n_tiles, tile_range(task, 1, G).n_tiles);
      for (int j = 0; j < n_tiles; ++j, ++it) {
        const int st = it % kStages, use = it / kStages;
        const int t0 = task.kv_begin + j * kTile;
        const int valid = min(kTile, task.kv_end - t0);
        const int npg = (valid + P - 1) / P;
        const uint32_t bytes = (uint32_t)(npg * KB) * box_bytes;
        const int pg = lane / KB, kb = lane % KB;
        const bool mine = lane < npg * KB;
        const int page = mine ? p.pages[task.page_off + (t0 + pg * P) / P] : 0;
        const uint32_t fb = smem_u32(&full[st]);
        if (!warp_wait(&empty[st], (use - 1) & 1, use > 0)) { fail(); ok = false; break; }
        if (lane == 0) mbar_expect_tx(fb, bytes);
        __syncwarp();
        if (mine)
          tma_load_4d(ring + st * Lay::kTileBytes + kb * 16384 + pg * P * 128, map, kb * 64, 0,
                      task.kv_head, page, fb);
      }
    }
    // every load this CTA started lands before it may exit
    if (lane == 0) {
      const uint64_t lim = ok ? 2000000000ull : 10000000ull;
      for (int j = (it > kStages ? it - kStages : 0); j < it; ++j) {
        const int st = j % kStages, use = j / kStages;
        mbar_wait(smem_u32(&full[st]), use & 1, lim);
      }
    }
  } else {
    // ------------------------------------------------------------- MMA issuer
    // The whole warp runs the loop (waits, the V-tail clear); one elected lane
    // issues the MMAs and commits.
    // The tensor core queues only a few MMAs and this warp shares its
    // scheduler with two busy softmax warps, so an MMA must cost the issuer
    // as few instructions as possible.  Each issue instance is compiled for a
    // fixed tile and stage; inside the elected branch the descriptors are the
    // stage's base descriptor plus the K step's constant offset, values the
    // compiler keeps uniform (holding all 48 descriptors in per-thread
    // registers made every MMA slower to issue), and no wait of this warp
    // reads the abort flag unless it has to block.
    constexpr uint32_t id_qk = idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t id_pv = idesc_bf16(128, D, 0, 1);
    constexpr int KS = D / 16;                      // K steps of QK
    constexpr int VS = kTile / 16;                  // K steps of PV
    uint32_t tS[2], tO[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      tS[x] = tm + x * 128;                         // S_x (P_x over its first 64 columns)
      tO[x] = tm + 256 + x * D;                     // O_x
    }
    // descriptor of K step ks: the base descriptor plus the step's offset / 16
    auto koff = [](int ks) { return (uint64_t)(((ks / 4) * 16384 + (ks % 4) * 32) >> 4); };
    int it = 0;                                     // KV tiles consumed (ring position)
    int px[2] = {0, 0};                             // phases consumed on p_full[X]
    int qn = 0;                                     // phases consumed on q_full
    bool ok = true;
    int t;
    using I0 = std::integral_constant<int, 0>;
    using I1 = std::integral_constant<int, 1>;
    auto qk_at = [&](auto xc, auto sc) {
      constexpr int X = decltype(xc)::value, ST = decltype(sc)::value;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t qd = smem_desc(q_base + X * Lay::kTileBytes, 16, 1024);
        const uint64_t kd = smem_desc(k_base + ST * Lay::kTileBytes, 16, 1024);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
          umma_ss(tS[X], qd + koff(ks), kd + koff(ks), id_qk, ks > 0);
        umma_commit(smem_u32(&bars.s_full[X]));
      }
      __syncwarp();
    };
    // O_X += P_X V over the first `steps` 16-key steps of the tile (a partial
    // tile's steps past its last key are skipped).
    auto pv_at = [&](auto xc, auto sc, int steps, bool first, bool last_of_task) {
      constexpr int X = decltype(xc)::value, ST = decltype(sc)::value;
      tc_fence_after();
      if (elect_one()) {
        const uint64_t vd = smem_desc(v_base + ST * Lay::kTileBytes, 16384, 1024);
        if (steps == VS && !first) {
#pragma unroll
          for (int ks = 0; ks < VS; ++ks) umma_ts(tO[X], tS[X] + ks * 8, vd + (uint64_t)(ks * 128), id_pv, 1u);
        } else {
#pragma unroll
          for (int ks = 0; ks < VS; ++ks)
            if (ks < steps)
              umma_ts(tO[X], tS[X] + ks * 8, vd + (uint64_t)(ks * 128), id_pv, (!first || ks > 0) ? 1u : 0u);
        }
        if (last_of_task) umma_commit(smem_u32(&bars.o_done[X]));
      }
      __syncwarp();
    };
    auto qk = [&](auto xc, int st) {
      if (st == 0) qk_at(xc, I0{}); else qk_at(xc, I1{});
    };
    auto pv = [&](auto xc, int st, int steps, bool first, bool last_of_task) {
      if (st == 0) pv_at(xc, I0{}, steps, first, last_of_task);
      else pv_at(xc, I1{}, steps, first, last_of_task);
    };
    // V rows past the task's last position inside its last 16-key step may
    // hold anything (NaN included); P is 0 there, and 0 * NaN would poison O,
    // so clear them (at most 15 rows).
    auto clear_v_tail = [&](int st, int valid) {
      uint8_t* vt = smem + Lay::v_off + st * Lay::kTileBytes;
      const int rows = ((valid + 15) & ~15) - valid;
      for (int idx = lane; idx < rows * 8 * KB; idx += 32) {
        const int kb = idx / (rows * 8);
        const int rem = idx - kb * rows * 8;
        *reinterpret_cast<int4*>(vt + kb * 16384 + (valid + rem / 8) * 128 + (rem % 8) * 16) =
            make_int4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      __syncwarp();
    };
    // one query tile's step of KV tile j: PV_X(j), then QK_X(j + 1) (V_j has
    // been waited for already)
    auto tile_step = [&](auto xc, int j, const int (&nt)[2], int st, int stn, int valid,
                         bool& k_ready) {
      constexpr int X = decltype(xc)::value;
      if (j >= nt[X]) return true;
      if (!warp_wait(&bars.p_full[X], px[X] & 1)) return false;
      ++px[X];
      pv(xc, st, (valid + 15) / 16, j == 0, j + 1 == nt[X]);
      if (j + 1 < nt[X]) {
        if (!k_ready) {
          if (!warp_wait(&bars.k_full[stn], ((it + j + 1) / kStages) & 1)) return false;
          k_ready = true;
        }
        qk(xc, stn);
      }
      return true;
    };
    for (int ti = 0; ok && (t = snake_task(ti, b, nctas)) < p.num_tasks; ++ti) {
      const pps::Task task = p.tasks[t];
      const int nt[2] = {tile_range(task, 0, G).n_tiles, tile_range(task, 1, G).n_tiles};
      const int n_tiles = max(nt[0], nt[1]);
      if (!warp_wait(&bars.q_full, qn & 1)) { fail(); ok = false; break; }
      ++qn;
      // QK of the first KV tile for both query tiles
      {
        const int st = it % kStages;
        if (!warp_wait(&bars.k_full[st], (it / kStages) & 1)) { fail(); ok = false; break; }
        if (nt[0] > 0) qk(I0{}, st);
        if (nt[1] > 0) qk(I1{}, st);
        tc_fence_after();
        if (elect_one()) umma_commit(smem_u32(&bars.k_empty[st]));   // K_0 used by both QKs
        __syncwarp();
      }
      // V_j is waited for (and its tail cleared) at the end of step j - 1, where
      // the wait's latency hides behind the MMAs just queued
      auto v_wait = [&](int j) -> bool {
        const int sj = (it + j) % kStages;
        if (!warp_wait(&bars.v_full[sj], ((it + j) / kStages) & 1)) return false;
        const int vj = min(kTile, task.kv_end - (task.kv_begin + j * kTile));
        if (vj & 15) clear_v_tail(sj, vj);
        return true;
      };
      if (n_tiles > 0 && !v_wait(0)) { fail(); ok = false; break; }
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int st = (it + j) % kStages;
        const int stn = (it + j + 1) % kStages;
        const bool next = j + 1 < n_tiles;
        const int valid = min(kTile, task.kv_end - (task.kv_begin + j * kTile));
        bool k_ready = false;
        if (!tile_step(I0{}, j, nt, st, stn, valid, k_ready) ||
            !tile_step(I1{}, j, nt, st, stn, valid, k_ready)) {
          fail();
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          umma_commit(smem_u32(&bars.v_empty[st]));                 // V_j no longer needed
          if (next) umma_commit(smem_u32(&bars.k_empty[stn]));      // K_{j+1} used by its QKs
        }
        __syncwarp();
        if (next && !v_wait(j + 1)) { fail(); ok = false; break; }
      }
      it += n_tiles;
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
    tmem_dealloc(tm, 512);
  }
}

template <int D>
int launch_t(const pps::Shape& s, const pps::DeviceTables& t, int64_t n, const void* q,
             const pps_pool& pool, void* out, int32_t* err, cudaStream_t st,
             const pps::AppendArgs* app) {
  CUtensorMap mk, mv;
  if (!pps::make_pool_map(&mk, pool.k, pool) || !pps::make_pool_map(&mv, pool.v, pool))
    return (int)cudaErrorInvalidValue;
  auto kern = mma_attention_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Layout<D>::smem_alloc);
  if (e != cudaSuccess) return (int)e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return (int)e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return (int)e;
  const int64_t grid = std::min<int64_t>(n, sms);
  MmaParams prm{t.mma_tasks, (int32_t)n, t.rows, t.pages, (const __nv_bfloat16*)q,
                (__nv_bfloat16*)out, t.o_part, t.lse_part, err, t.tree_mask, s.num_q_heads, s.group,
                s.page_size, s.sm_scale * 1.4426950408889634f,
                app ? *app : pps::AppendArgs{}, pool.k, pool.v, pool.num_kv_heads,
                pool.num_pages, t.sync};
  // with the append every CTA must be resident at once (it waits for all)
  e = app ? pps::launch_cooperative(kern, (unsigned)grid, kThreads, Layout<D>::smem_alloc, st, mk,
                                    mv, prm)
          : pps::launch_dependent(kern, (unsigned)grid, kThreads, Layout<D>::smem_alloc, st, mk, mv,
                                  prm);
  pps::count_launch();
  return (int)e;
}

}  // namespace

namespace pps {

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
  // Encoding a map is host work on every launch; a serving loop reuses the
  // same pool arrays, so the last few maps are kept (keyed by every field the
  // encoding reads).
  struct Entry {
    const void* base;
    int32_t D, P, H, pages;
    CUtensorMap map;
  };
  static std::mutex mu;
  static Entry cache[8];
  static int used = 0, next = 0;
  const int D = pool.head_dim, P = pool.page_size, H = pool.num_kv_heads;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < used; ++i) {
      const Entry& e = cache[i];
      if (e.base == base && e.D == D && e.P == P && e.H == H && e.pages == pool.num_pages) {
        *map = e.map;
        return true;
      }
    }
  }
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)P, (cuuint64_t)H, (cuuint64_t)pool.num_pages};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)P * D * 2, (cuuint64_t)H * P * D * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)P, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  if (fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lk(mu);
  cache[next] = Entry{base, D, P, H, pool.num_pages, *map};
  next = (next + 1) % 8;
  used = used < 8 ? used + 1 : 8;
  return true;
}

bool mma_path_available() { return true; }

int launch_mma_attention(const Shape& s, const DeviceTables& t, int64_t num_tasks, const void* q,
                         const pps_pool& pool, void* out, int32_t* err, void* stream,
                         const AppendArgs* app) {
  if (num_tasks == 0) return cudaSuccess;
  auto st = (cudaStream_t)stream;
  if (s.head_dim == 128) return launch_t<128>(s, t, num_tasks, q, pool, out, err, st, app);
  return launch_t<64>(s, t, num_tasks, q, pool, out, err, st, app);
}

}  // namespace pps
