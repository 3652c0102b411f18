// Host tile planner: turns one mixed prefill/decode/verify batch into a
// work-sorted task table (pps_attn_plan, pps_attn_plan_tree).
//
// Follows the XY-Serve review (pith.science/paper/ABCKJ6RF): "Core claim"
// (every stage's attention decomposed into tile tasks recorded in tables),
// "What carries the argument" (tiles sorted by computational area before they
// are handed to cores), and the SGLang review (pith.science/p/2312.07104),
// "Core claim" (RadixAttention: requests that share a cached prefix share its
// KV).  Shared runs of pages are found with a radix tree over page ids, built
// here from the lexicographically sorted page lists and their longest common
// prefixes.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <numeric>
#include <unordered_map>

#include "pps_internal.h"

namespace {

using pps::Task;

// Per-thread page stamps reused across calls (no per-plan allocation of a
// pool-sized array): entry p is "set in this pass" when it equals the pass's
// epoch.
thread_local std::vector<uint32_t> g_page_stamp;
thread_local uint32_t g_epoch = 0;
uint32_t next_epoch(int32_t num_pages) {
  if (g_page_stamp.size() < (size_t)num_pages) {
    g_page_stamp.assign((size_t)num_pages, 0);
    g_epoch = 0;
  }
  if (++g_epoch == 0) {                       // wrapped: start over
    std::fill(g_page_stamp.begin(), g_page_stamp.end(), 0);
    g_epoch = 1;
  }
  return g_epoch;
}

struct Segment {       // KV positions [kv_begin, kv_end) of one page list, with query tokens
  int32_t row_off;     // first token in the rows array
  int32_t n_tok;
  int32_t page_off;
  int32_t kv_begin, kv_end;
  bool causal;         // private segment: token i sees positions <= c + i
  int32_t c;
  int32_t key;         // request id (private) or R + group id (group), for stable ordering
};

struct TaskSet {       // emitted once per kv head
  int32_t row_off, n_tok, page_off, kv_begin, kv_end, causal;
  int32_t key, tile, chunk;
  bool mma;
  int64_t work;
  int32_t out_pid;
};

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Pages two sequences share from the start (first n at most), compared in
// 32-byte blocks.
inline int32_t common_pages(const int32_t* a, const int32_t* b, int32_t n) {
  int32_t k = 0;
  while (k + 8 <= n && std::memcmp(a + k, b + k, 32) == 0) k += 8;
  while (k < n && a[k] == b[k]) ++k;
  return k;
}

bool pow2_in(int32_t v, std::initializer_list<int32_t> set) {
  for (int32_t s : set) if (v == s) return true;
  return false;
}

// Radix tree over page-id sequences: requests sorted lexicographically by their
// fully cached page lists; lcp[i] = common prefix (in pages) of sorted[i-1] and
// sorted[i].  Every maximal run sharing more than `depth` pages is a node.
struct RadixBuilder {
  const std::vector<int32_t>& sorted;
  const std::vector<int32_t>& lcp;
  std::vector<std::pair<std::vector<int32_t>, std::pair<int32_t, int32_t>>> groups;  // members, [d0, d1)
  std::vector<int32_t>& group_end;  // per request: deepest grouped page

  void build(int32_t lo, int32_t hi, int32_t depth) {
    int32_t i = lo;
    while (i < hi) {
      int32_t j = i + 1;
      int32_t common = INT32_MAX;
      while (j < hi && lcp[j] > depth) {
        common = std::min(common, lcp[j]);
        ++j;
      }
      if (j - i >= 2) {
        std::vector<int32_t> members(sorted.begin() + i, sorted.begin() + j);
        std::sort(members.begin(), members.end());
        for (int32_t r : members) group_end[r] = std::max(group_end[r], common);
        groups.push_back({std::move(members), {depth, common}});
        build(i, j, common);
      }
      i = j;
    }
  }
};

}  // namespace

extern "C" pps_status pps_attn_plan(const int32_t* q_indptr, const int32_t* kv_len,
                                    const int32_t* page_indptr, const int32_t* page_indices,
                                    int32_t num_requests, int32_t num_q_heads,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                                    int32_t num_pages, float sm_scale,
                                    const pps_plan_options* opts, pps_plan** out_plan,
                                    size_t* out_workspace_bytes) {
  return pps_attn_plan_tree(q_indptr, kv_len, page_indptr, page_indices, nullptr, num_requests,
                            num_q_heads, num_kv_heads, head_dim, page_size, num_pages, sm_scale,
                            opts, out_plan, out_workspace_bytes);
}

extern "C" pps_status pps_attn_plan_tree(const int32_t* q_indptr, const int32_t* kv_len,
                                         const int32_t* page_indptr, const int32_t* page_indices,
                                         const int32_t* tree_parent, int32_t num_requests,
                                         int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t page_size, int32_t num_pages,
                                         float sm_scale, const pps_plan_options* opts,
                                         pps_plan** out_plan, size_t* out_workspace_bytes) {
  return pps::plan_tree(q_indptr, kv_len, page_indptr, page_indices, tree_parent, num_requests,
                        num_q_heads, num_kv_heads, head_dim, page_size, num_pages, sm_scale, opts,
                        0, out_plan, out_workspace_bytes);
}

pps_status pps::plan_tree(const int32_t* q_indptr, const int32_t* kv_len,
                          const int32_t* page_indptr, const int32_t* page_indices,
                          const int32_t* tree_parent, int32_t num_requests, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                          int32_t num_pages, float sm_scale, const pps_plan_options* opts,
                          int32_t split_request, pps_plan** out_plan,
                          size_t* out_workspace_bytes) {
  if (out_plan) *out_plan = nullptr;
  if (out_workspace_bytes) *out_workspace_bytes = 0;
  if (!out_plan || !out_workspace_bytes || num_requests < 0 || !q_indptr || !page_indptr ||
      (num_requests > 0 && !kv_len) || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_pages < 0 || !std::isfinite(sm_scale))
    return PPS_ERR_INVALID_ARGUMENT;
  if (num_q_heads % num_kv_heads) return PPS_ERR_INVALID_ARGUMENT;
  const int32_t G = num_q_heads / num_kv_heads;
  if (!pow2_in(G, {1, 2, 4, 8}) || !pow2_in(head_dim, {64, 128}) ||
      !pow2_in(page_size, {16, 32, 64, 128}))
    return PPS_ERR_UNSUPPORTED;
  const int32_t R = num_requests, P = page_size;
  if (q_indptr[0] != 0 || page_indptr[0] != 0) return PPS_ERR_INVALID_ARGUMENT;
  for (int32_t r = 0; r < R; ++r) {
    if (q_indptr[r + 1] < q_indptr[r]) return PPS_ERR_INVALID_ARGUMENT;
    if (page_indptr[r + 1] < page_indptr[r]) return PPS_ERR_PAGE_TABLE;
    const int32_t q = q_indptr[r + 1] - q_indptr[r];
    if (kv_len[r] < q) return PPS_ERR_INVALID_ARGUMENT;
    const int64_t need = ceil_div(kv_len[r], P);
    if (page_indptr[r + 1] - page_indptr[r] < need) return PPS_ERR_PAGE_TABLE;
    // ids in [0, num_pages): one unsigned compare per id, OR-ed without
    // branches so the loop vectorizes
    const int32_t* pl = page_indices + page_indptr[r];
    uint32_t bad = 0;
    for (int64_t i = 0; i < need; ++i) bad |= (uint32_t)((uint32_t)pl[i] >= (uint32_t)num_pages);
    if (bad) return PPS_ERR_PAGE_TABLE;
  }
  const int64_t nnz = page_indptr[R];
  if (nnz > 0 && !page_indices) return PPS_ERR_INVALID_ARGUMENT;
  // Draft trees: parents precede their children; a request whose parents are
  // not the chain j - 1 is a tree and must fit the 64-bit per-token mask.
  int32_t num_tree = 0;
  if (tree_parent) {
    for (int32_t r = 0; r < R; ++r) {
      const int32_t t0 = q_indptr[r], q = q_indptr[r + 1] - t0;
      bool chain = true;
      for (int32_t j = 0; j < q; ++j) {
        const int32_t a = tree_parent[t0 + j];
        if (a < -1 || a >= j) return PPS_ERR_INVALID_ARGUMENT;
        chain &= (a == j - 1);
      }
      if (!chain) {
        if (q > PPS_TREE_MAX_TOKENS) return PPS_ERR_UNSUPPORTED;
        ++num_tree;
      }
    }
  }

  pps_plan_options o{};
  if (opts) o = *opts;
  int32_t num_sms = o.num_sms;
  if (num_sms <= 0) num_sms = pps::device_sm_count();
  if (num_sms <= 0) num_sms = 152;
  const bool use_mma = pps::mma_path_available() && !(o.flags & PPS_PLAN_CUDA_CORES_ONLY);
  const bool use_groups = !(o.flags & PPS_PLAN_NO_GROUPS);

  pps_plan* plan = new (std::nothrow) pps_plan;
  if (!plan) return PPS_ERR_NO_MEMORY;
  try {
    plan->shape = {num_q_heads, num_kv_heads, head_dim, page_size, G, num_pages, sm_scale, 0, 0, 0};
    plan->num_requests = R;
    plan->num_tokens = q_indptr[R];
    plan->use_mma = use_mma;
    const int32_t T = q_indptr[R];
    plan->num_tree_requests = num_tree;
    plan->has_tree = num_tree > 0;

    // ---- 0. per-token lookback masks of draft trees -----------------------------------
    // anc = ancestor-or-self set over the request's new-token indices (bit i =
    // token i); lookback bit k = visibility of the key k positions back, which
    // for k <= j is new token j - k, and a cached position beyond that.
    std::vector<uint64_t> tmask;
    if (plan->has_tree) {
      tmask.assign((size_t)T, ~0ull);
      std::vector<uint64_t> anc;
      for (int32_t r = 0; r < R; ++r) {
        const int32_t t0 = q_indptr[r], q = q_indptr[r + 1] - t0;
        bool chain = true;
        for (int32_t j = 0; j < q; ++j) chain &= (tree_parent[t0 + j] == j - 1);
        if (chain) continue;
        anc.assign((size_t)q, 0);
        for (int32_t j = 0; j < q; ++j) {
          const int32_t a = tree_parent[t0 + j];
          anc[j] = (1ull << j) | (a >= 0 ? anc[a] : 0ull);
          uint64_t m = ~0ull;
          for (int32_t k = 0; k <= j; ++k)
            if (!((anc[j] >> (j - k)) & 1ull)) m &= ~(1ull << k);
          tmask[t0 + j] = m;
        }
      }
    }

    // ---- 1. radix grouping over fully cached pages --------------------------------
    // A request joins the grouping when its rows fill at most half a
    // tensor-core tile.  A group saves shared-page reads only by packing the
    // rows of several requests into fewer tiles; each grouped token pays fp32
    // partials (~1 KB per query head, written and merged).  Decode and verify
    // rows gain most; a prefill chunk of whole tiles gains nothing, so it reads
    // the shared pages in its own tiles and writes its rows directly.  Plans
    // without tensor-core tiles (16-row CUDA-core tiles) group every request.
    std::vector<int32_t> group_end(R, 0);
    std::vector<std::pair<std::vector<int32_t>, std::pair<int32_t, int32_t>>> groups;
    if (use_groups) {
      const int64_t max_rows = use_mma ? pps::kMmaTaskRows / 2 : INT64_MAX;
      std::vector<int32_t> full(R, 0), cand;
      for (int32_t r = 0; r < R; ++r) {
        const int32_t q = q_indptr[r + 1] - q_indptr[r];
        const int32_t c = kv_len[r] - q;
        full[r] = c / P;
        if (q > 0 && full[r] > 0 && (int64_t)q * G <= max_rows) cand.push_back(r);
      }
      auto seq = [&](int32_t r) { return page_indices + page_indptr[r]; };
      // A group needs two requests whose first cached pages are the same; with
      // none, the sort below has nothing to find.
      {
        uint32_t ep = next_epoch(num_pages);
        uint32_t* stamp = g_page_stamp.data();     // thread-local lookups hoisted
        bool any = false;
        for (int32_t r : cand) {
          uint32_t& m = stamp[seq(r)[0]];
          if (m == ep) { any = true; break; }
          m = ep;
        }
        if (!any) cand.clear();
      }
      // A lexicographic order of the page lists (page ids compared as their
      // 4 bytes in memory order, one memcmp over the common length): every set
      // of lists sharing a prefix is then one contiguous run.
      std::sort(cand.begin(), cand.end(), [&](int32_t a, int32_t b) {
        const int32_t n = std::min(full[a], full[b]);
        const int c = std::memcmp(seq(a), seq(b), (size_t)n * 4);
        if (c != 0) return c < 0;
        if (full[a] != full[b]) return full[a] < full[b];
        return a < b;
      });
      std::vector<int32_t> lcp(cand.size(), 0);
      for (size_t i = 1; i < cand.size(); ++i) {
        const int32_t a = cand[i - 1], b = cand[i];
        lcp[i] = common_pages(seq(a), seq(b), std::min(full[a], full[b]));
      }
      RadixBuilder rb{cand, lcp, {}, group_end};
      rb.build(0, (int32_t)cand.size(), 0);
      groups = std::move(rb.groups);
    }
    plan->num_groups = (int32_t)groups.size();

    // ---- 2. segments ---------------------------------------------------------------
    std::vector<int32_t> rows;
    rows.reserve((size_t)T * 2);
    std::vector<Segment> segs;
    for (size_t g = 0; g < groups.size(); ++g) {
      const auto& mem = groups[g].first;
      Segment s{};
      s.row_off = (int32_t)rows.size();
      for (int32_t r : mem)
        for (int32_t t = q_indptr[r]; t < q_indptr[r + 1]; ++t) rows.push_back(t);
      s.n_tok = (int32_t)rows.size() - s.row_off;
      s.page_off = page_indptr[mem[0]];
      s.kv_begin = groups[g].second.first * P;
      s.kv_end = groups[g].second.second * P;
      s.causal = false;
      s.c = 0;
      s.key = R + (int32_t)g;
      segs.push_back(s);
    }
    for (int32_t r = 0; r < R; ++r) {
      const int32_t q = q_indptr[r + 1] - q_indptr[r];
      if (q == 0) continue;
      Segment s{};
      s.row_off = (int32_t)rows.size();
      for (int32_t t = q_indptr[r]; t < q_indptr[r + 1]; ++t) rows.push_back(t);
      s.n_tok = q;
      s.page_off = page_indptr[r];
      s.kv_begin = group_end[r] * P;
      s.kv_end = kv_len[r];
      s.causal = true;
      s.c = kv_len[r] - q;
      s.key = r;
      segs.push_back(s);
    }

    // ---- 3. tiles and split-KV chunks ----------------------------------------------
    // Small-row tasks (decode tokens, short drafts and draft trees, narrow
    // shared-prefix groups): up to 32 rows on the key-tile tensor kernel
    // (head_dim 128), else up to 8 rows on the CUDA-core kernel.
    const bool use_tt = use_mma && head_dim == 128 && G <= pps::kTtRows &&
                        !(o.flags & PPS_PLAN_SMALL_ROWS_CUDA_CORES);
    plan->shape.small_tt = use_tt ? 1 : 0;
    const int32_t bw_max_tok = use_tt ? pps::kTtRows / G : std::max(1, 8 / G);
    const int32_t bw_tile_tok = std::max(1, pps::kBwMaxRows / G);
    const int32_t mma_tile_tok = pps::kMmaTaskRows / G;
    auto is_mma = [&](const Segment& s) { return use_mma && s.n_tok > bw_max_tok; };
    auto tile_tok_of = [&](const Segment& s) {
      if (is_mma(s)) return mma_tile_tok;
      return s.n_tok <= bw_max_tok ? s.n_tok : bw_tile_tok;
    };
    // Spans before chunking: [a, b) split into chunks; the last chunk runs to `end`.
    struct Span { int32_t a, b, end; };
    auto span_of = [&](const Segment& s, int32_t i0, int32_t i1) {
      if (!s.causal) return Span{s.kv_begin, s.kv_end, s.kv_end};
      return Span{s.kv_begin, s.c + i0 + 1, std::min(s.kv_end, s.c + i1)};
    };
    int64_t bw_kv = 0, mma_kv = 0, mma_tiles = 0;
    for (const auto& s : segs) {
      const int32_t tt = tile_tok_of(s);
      for (int32_t i0 = 0; i0 < s.n_tok; i0 += tt) {
        const Span sp = span_of(s, i0, std::min(s.n_tok, i0 + tt));
        if (is_mma(s)) { mma_kv += sp.end - sp.a; ++mma_tiles; }
        else bw_kv += sp.end - sp.a;
      }
    }
    // The small-row kernels are persistent (one CTA per SM; the CUDA-core one
    // takes the work-sorted tasks in symmetric round-robin order, the key-tile
    // one its per-CTA range), so tasks only need to be small enough to give
    // every SM about two of them: each task costs a
    // query load and a cross-warp merge, and a split request costs partials
    // and a merge.  Measured on GB300: 4096-token tasks beat 2048 (decode,
    // 256 requests) and 1024+ beat 352 (radix subtrees, 64 requests).
    int32_t bw_chunk = o.bw_chunk_tokens;
    if (bw_chunk <= 0) {
      const int64_t want = ceil_div(bw_kv * num_kv_heads, (int64_t)num_sms * 2);
      bw_chunk = (int32_t)std::min<int64_t>(4096, std::max<int64_t>(128, want));
    }
    {
      const int32_t unit = use_tt ? pps::kMmaKvTile : P;   // whole 128-key tiles on tensor cores
      bw_chunk = (int32_t)(ceil_div(bw_chunk, unit) * unit);
    }
    int32_t mma_chunk = o.mma_chunk_tokens;
    if (mma_chunk <= 0) {
      mma_chunk = 1 << 30;
      const int64_t target = 2LL * num_sms;
      if (mma_tiles * num_kv_heads > 0 && mma_tiles * num_kv_heads < target) {
        const int64_t want = ceil_div(mma_kv * num_kv_heads, target);
        mma_chunk = (int32_t)std::max<int64_t>(512, want);
      }
    }
    mma_chunk = (int32_t)std::min<int64_t>(1 << 30, ceil_div(mma_chunk, pps::kMmaKvTile) * pps::kMmaKvTile);

    std::vector<TaskSet> sets;
    for (const auto& s : segs) {
      const bool mma = is_mma(s);
      const int32_t tt = tile_tok_of(s);
      const int32_t chunk = mma ? mma_chunk : bw_chunk;
      int32_t tile = 0;
      for (int32_t i0 = 0; i0 < s.n_tok; i0 += tt, ++tile) {
        const int32_t i1 = std::min(s.n_tok, i0 + tt);
        const Span sp = span_of(s, i0, i1);
        int64_t step = chunk;
        int64_t nch = std::max<int64_t>(1, ceil_div(sp.b - sp.a, chunk));
        if (!mma && use_tt && o.bw_chunk_tokens <= 0) {
          // key-tile tasks: no split within a quarter over the chunk, else
          // equal whole-tile pieces (no one-tile remainder task)
          const int64_t span = sp.b - sp.a;
          nch = span <= chunk + chunk / 4 ? 1 : ceil_div(span, chunk);
          step = ceil_div(ceil_div(span, nch), pps::kMmaKvTile) * pps::kMmaKvTile;
          nch = std::max<int64_t>(1, ceil_div(span, step));
        }
        for (int64_t k = 0; k < nch; ++k) {
          TaskSet ts{};
          ts.row_off = s.row_off + i0;
          ts.n_tok = i1 - i0;
          ts.page_off = s.page_off;
          ts.kv_begin = sp.a + (int32_t)(k * step);
          ts.kv_end = (k == nch - 1) ? sp.end : ts.kv_begin + (int32_t)step;
          ts.causal = s.causal ? s.c + i0 : PPS_NO_CAUSAL;
          ts.key = s.key;
          ts.tile = tile;
          ts.chunk = (int32_t)k;
          ts.mma = mma;
          if (!mma && use_tt) {
            // key-tile tasks stream K/V at the memory rate whatever their rows:
            // time ~ 128-key tiles, plus about two tiles of per-task work
            ts.work = (ceil_div(ts.kv_end - ts.kv_begin, pps::kMmaKvTile) + 2) * pps::kMmaKvTile;
          } else {
            const int64_t rows_eff = mma ? pps::kMmaTaskRows : (int64_t)ts.n_tok * G;
            ts.work = rows_eff * (ts.kv_end - ts.kv_begin);
          }
          ts.out_pid = -1;
          sets.push_back(ts);
        }
      }
    }

    // ---- 4. partial slots and merge lists ------------------------------------------
    // A task set writes its rows directly when each of its tokens is covered by
    // this set alone; otherwise every token of the set gets a partial slot, and
    // the merge lists (CSR over the tokens in increasing order, slots in task
    // order) name them.  Built in three passes over flat arrays.
    std::vector<int32_t> pieces(T, 0);
    for (const auto& ts : sets)
      for (int32_t i = 0; i < ts.n_tok; ++i) ++pieces[rows[ts.row_off + i]];
    std::vector<uint8_t> direct(sets.size(), 1);
    std::vector<int32_t> slots(T + 1, 0);             // partial slots per token, then offsets
    for (size_t k = 0; k < sets.size(); ++k) {
      const auto& ts = sets[k];
      for (int32_t i = 0; i < ts.n_tok; ++i)
        if (pieces[rows[ts.row_off + i]] != 1) { direct[k] = 0; break; }
      if (!direct[k])
        for (int32_t i = 0; i < ts.n_tok; ++i) ++slots[rows[ts.row_off + i] + 1];
    }
    std::vector<int32_t> m_tok, m_ptr{0}, m_pid;
    std::vector<int32_t> first(T, 0);                 // token -> first slot in m_pid
    for (int32_t t = 0; t < T; ++t) {
      if (!slots[t + 1]) continue;
      first[t] = m_ptr.back();
      m_tok.push_back(t);
      m_ptr.push_back(m_ptr.back() + slots[t + 1]);
    }
    m_pid.resize((size_t)m_ptr.back());
    std::fill(slots.begin(), slots.end(), 0);         // now: slots filled per token
    int64_t next_pid = 0;
    for (size_t k = 0; k < sets.size(); ++k) {
      auto& ts = sets[k];
      if (direct[k]) continue;
      ts.out_pid = (int32_t)next_pid;
      for (int32_t i = 0; i < ts.n_tok; ++i) {
        const int32_t t = rows[ts.row_off + i];
        m_pid[first[t] + slots[t]++] = (int32_t)(next_pid + i);
      }
      next_pid += ts.n_tok;
    }

    // ---- 5. sort by work (descending), deterministic ties ---------------------------
    // Order: bandwidth before tensor-core sets, then work descending, then
    // (key, tile, chunk), which identify a set, so the order is total.  A
    // split request puts the tensor-core sets of the requests before it first
    // (each half in work order), when the split can hold: tensor-core sets
    // only, every one private to a request (no shared-prefix group), no
    // partials.
    bool split = split_request > 0 && split_request < R;
    for (size_t k = 0; split && k < sets.size(); ++k)
      split = sets[k].mma && sets[k].key < R && direct[k];
    {
      struct SortKey {
        uint64_t a, b;
        uint32_t c, idx;
      };
      std::vector<SortKey> keys(sets.size());
      for (size_t k = 0; k < sets.size(); ++k) {
        const TaskSet& t = sets[k];
        const uint64_t late = split && t.key >= split_request ? 1 : 0;
        keys[k].a = ((uint64_t)t.mma << 63) | (late << 62) |
                    (((uint64_t)1 << 61) - 1 - (uint64_t)t.work);
        keys[k].b = ((uint64_t)(uint32_t)t.key << 32) | (uint32_t)t.tile;
        keys[k].c = (uint32_t)t.chunk;
        keys[k].idx = (uint32_t)k;
      }
      std::sort(keys.begin(), keys.end(), [](const SortKey& x, const SortKey& y) {
        if (x.a != y.a) return x.a < y.a;
        if (x.b != y.b) return x.b < y.b;
        return x.c < y.c;
      });
      std::vector<TaskSet> sorted(sets.size());
      for (size_t k = 0; k < sets.size(); ++k) sorted[k] = sets[keys[k].idx];
      sets.swap(sorted);
    }
    std::vector<Task> bw, mm;
    {
      size_t n_mma = 0;
      for (const auto& ts : sets) n_mma += ts.mma ? 1 : 0;
      bw.reserve((sets.size() - n_mma) * (size_t)num_kv_heads);
      mm.reserve(n_mma * (size_t)num_kv_heads);
    }
    for (const auto& ts : sets) {
      if (!ts.mma) plan->shape.bw_rows_max = std::max(plan->shape.bw_rows_max, ts.n_tok * G);
      for (int32_t h = 0; h < num_kv_heads; ++h) {
        Task t{ts.row_off, ts.n_tok, h, ts.page_off, ts.kv_begin, ts.kv_end, ts.causal, ts.out_pid};
        (ts.mma ? mm : bw).push_back(t);
      }
    }
    // Key-tile plans: the persistent kernel's CTAs take contiguous ranges of
    // the table.  Each task, largest first, goes to a CTA with the least work
    // so far, and keeps that order inside its range: tt_cta[b] .. tt_cta[b + 1]
    // for CTA b.  The work unit is the key-tile kernel's: whole 128-key tiles
    // plus two for the task's own work.  Loads are small integers that only
    // grow, so the CTAs sit in buckets by load (first in, first out: ties go
    // to the CTA that reached the load first, CTA order at the start) and the
    // lowest non-empty bucket only moves up: O(tasks + buckets).
    std::vector<int32_t> tt_cta, owner;     // owner: CTA of each bw task (scattered at 7.)
    if (use_tt && !bw.empty()) {
      const int32_t C = (int32_t)std::min<int64_t>((int64_t)bw.size(), num_sms);
      std::vector<int32_t> w(bw.size());
      int64_t total = 0, wmax = 0;
      for (size_t k = 0; k < bw.size(); ++k) {
        w[k] = (int32_t)ceil_div(bw[k].kv_end - bw[k].kv_begin, pps::kMmaKvTile) + 2;
        total += w[k];
        wmax = std::max<int64_t>(wmax, w[k]);
      }
      // a CTA is picked at the least load (at most the mean), so every load
      // stays below total / C + wmax + 1
      const size_t nb = (size_t)(total / C + wmax + 2);
      std::vector<int32_t> first(nb, -1), last(nb, -1), next((size_t)C, -1);
      for (int32_t b = 0; b < C; ++b) next[b] = b + 1 < C ? b + 1 : -1;
      first[0] = 0;
      last[0] = C - 1;
      owner.resize(bw.size());
      tt_cta.assign((size_t)C + 1, 0);
      size_t cur = 0;
      for (size_t k = 0; k < bw.size(); ++k) {
        while (first[cur] < 0) ++cur;
        const int32_t b = first[cur];
        first[cur] = next[b];
        if (first[cur] < 0) last[cur] = -1;
        owner[k] = b;
        ++tt_cta[(size_t)b + 1];
        const size_t to = cur + (size_t)w[k];
        next[b] = -1;
        if (last[to] < 0) first[to] = b;
        else next[last[to]] = b;
        last[to] = b;
      }
      for (int32_t b = 0; b < C; ++b) tt_cta[(size_t)b + 1] += tt_cta[b];
    }
    plan->shape.tt_ctas = tt_cta.empty() ? 0 : (int32_t)tt_cta.size() - 1;

    // ---- 6. statistics ---------------------------------------------------------------
    const int64_t tok_bytes = 2LL * num_kv_heads * head_dim * 2;   // K+V, all kv heads
    {
      // the unique-slot count runs on demand (pps_plan_get_info) from these
      plan->kv_len_copy.assign(kv_len, kv_len + R);
      plan->page_indptr_copy.assign(page_indptr, page_indptr + R + 1);
      plan->tok_bytes = tok_bytes;

    }
    double fl_tot = 0, fl_mma = 0;
    int64_t read = 0, read_bw = 0;
    double issued = 0;
    for (const auto& ts : sets) {
      double pairs = 0;
      for (int32_t i = 0; i < ts.n_tok; ++i) {
        const int64_t lim = std::min<int64_t>(ts.kv_end, (int64_t)ts.causal + i + 1);
        pairs += (double)std::max<int64_t>(0, lim - ts.kv_begin);
        if (plan->has_tree && ts.causal != PPS_NO_CAUSAL) {
          const uint64_t m = tmask[rows[ts.row_off + i]];
          for (int k = 0; k < 64 && m != ~0ull; ++k) {
            const int64_t pos = (int64_t)ts.causal + i - k;
            if (!((m >> k) & 1ull) && pos >= ts.kv_begin && pos < lim) pairs -= 1;
          }
        }
      }
      const double f = pairs * num_q_heads * 4.0 * head_dim;
      fl_tot += f;
      if (ts.mma) fl_mma += f;
      read += (int64_t)(ts.kv_end - ts.kv_begin) * tok_bytes;
      if (!ts.mma) {
        read_bw += (int64_t)(ts.kv_end - ts.kv_begin) * tok_bytes;
        if (use_tt)   // 128 keys x 32 rows x d per tile and kv head
          issued += (double)ceil_div(ts.kv_end - ts.kv_begin, pps::kMmaKvTile) * num_kv_heads *
                    4.0 * pps::kMmaKvTile * pps::kTtRows * head_dim;
      } else {
        // whole tiles per kv head: ceil(rows / 128) x ceil(span / 128) of 128 x 128 x d
        const int64_t tiles = ceil_div((int64_t)ts.n_tok * G, pps::kMmaRows) *
                              ceil_div(ts.kv_end - ts.kv_begin, pps::kMmaKvTile);
        issued += (double)tiles * num_kv_heads * 4.0 * pps::kMmaRows * pps::kMmaKvTile * head_dim;
      }
    }
    plan->flops_total = fl_tot;
    plan->flops_mma = fl_mma;
    plan->kv_bytes_read = read;
    plan->kv_bytes_bw = read_bw;
    plan->flops_mma_issued = issued;

    // ---- 7. table image ----------------------------------------------------------------
    auto al = [](int64_t n) { return (n + 63) / 64 * 64; };
    pps::TableLayout L;
    int64_t off = 0;
    L.bw_tasks = off;      off += al((int64_t)bw.size() * PPS_TASK_INTS);
    L.mma_tasks = off;     off += al((int64_t)mm.size() * PPS_TASK_INTS);
    L.rows = off;          off += al((int64_t)rows.size());
    L.pages = off;         off += al(nnz);
    L.merge_tokens = off;  off += al((int64_t)m_tok.size());
    L.merge_indptr = off;  off += al((int64_t)m_ptr.size());
    L.merge_pids = off;    off += al((int64_t)m_pid.size());
    L.tree_mask = off;     off += plan->has_tree ? al(2LL * T) : 0;
    L.tt_cta = off;        off += al((int64_t)tt_cta.size());
    L.sync = off;          off += 64;             // zeros: a counter for grid-wide waits
    L.total_ints = off;
    plan->layout = L;
    plan->image_ints = std::max<int64_t>(off, 64);
    plan->image = pps::host_buf_acquire((size_t)plan->image_ints);
    if (!plan->image.data) throw std::bad_alloc();
    int32_t* img = plan->image.data;
    // Each section is copied in (src null: already written) and the alignment
    // gap after it zeroed.
    auto put = [&](int64_t at, const void* src, int64_t ints, int64_t end) {
      if (ints && src) std::memcpy(img + at, src, (size_t)ints * 4);
      if (end > at + ints) std::memset(img + at + ints, 0, (size_t)(end - at - ints) * 4);
    };
    if (owner.empty()) {
      put(L.bw_tasks, bw.data(), (int64_t)bw.size() * PPS_TASK_INTS, L.mma_tasks);
    } else {                 // key-tile tables: each task at its place in its CTA's range
      std::vector<int32_t> at(tt_cta.begin(), tt_cta.end() - 1);
      Task* dst = reinterpret_cast<Task*>(img + L.bw_tasks);
      for (size_t k = 0; k < bw.size(); ++k) dst[at[owner[k]]++] = bw[k];
      put(L.bw_tasks, nullptr, (int64_t)bw.size() * PPS_TASK_INTS, L.mma_tasks);
    }
    put(L.mma_tasks, mm.data(), (int64_t)mm.size() * PPS_TASK_INTS, L.rows);
    put(L.rows, rows.data(), (int64_t)rows.size(), L.pages);
    put(L.pages, page_indices, nnz, L.merge_tokens);
    put(L.merge_tokens, m_tok.data(), (int64_t)m_tok.size(), L.merge_indptr);
    put(L.merge_indptr, m_ptr.data(), (int64_t)m_ptr.size(), L.merge_pids);
    put(L.merge_pids, m_pid.data(), (int64_t)m_pid.size(), L.tree_mask);
    put(L.tree_mask, tmask.data(), plan->has_tree ? 2LL * T : 0, L.tt_cta);
    put(L.tt_cta, tt_cta.data(), (int64_t)tt_cta.size(), L.sync);
    put(L.sync, nullptr, 0, plan->image_ints);

    plan->num_bw = (int64_t)bw.size();
    plan->num_mma = (int64_t)mm.size();
    if (split) {
      int64_t first = 0;
      for (const auto& ts : sets) first += ts.key < split_request ? num_kv_heads : 0;
      if (first > 0 && first < plan->num_mma) {
        plan->num_mma_first = first;
        plan->split_tokens = q_indptr[split_request];
      }
    }
    plan->num_partials = next_pid;
    plan->num_merge_tokens = (int64_t)m_tok.size();
    plan->num_merge_pids = (int64_t)m_pid.size();
    plan->num_rows = (int64_t)rows.size();
    plan->num_pages_listed = nnz;
    auto al256 = [](size_t n) { return (n + 255) / 256 * 256; };
    plan->table_bytes = al256((size_t)plan->image_ints * 4);
    plan->partial_o_bytes = al256((size_t)next_pid * num_q_heads * head_dim * 4);
    plan->partial_lse_bytes = al256((size_t)next_pid * num_q_heads * 4);
    plan->workspace_bytes = plan->table_bytes + plan->partial_o_bytes + plan->partial_lse_bytes;
  } catch (const std::bad_alloc&) {
    delete plan;
    return PPS_ERR_NO_MEMORY;
  }
  *out_plan = plan;
  *out_workspace_bytes = plan->workspace_bytes;
  return PPS_OK;
}

extern "C" pps_status pps_plan_destroy(pps_plan* plan) {
  delete plan;
  return PPS_OK;
}

namespace {
// K+V bytes of the distinct (page, kv head, valid slot) triples of a plan's
// requests: valid slots counted per page (P <= 128 fits a byte); every page of
// a request is full but its last, and the update is branch-free.
int64_t unique_kv_bytes(const pps_plan* p) {
  const int32_t P = p->shape.page_size, R = p->num_requests;
  const int32_t* pages = p->image.data + p->layout.pages;
  std::vector<uint8_t> seen((size_t)p->shape.num_pages, 0);
  int64_t slots = 0;
  for (int32_t r = 0; r < R; ++r) {
    const int32_t kv = p->kv_len_copy[r];
    const int32_t need = (int32_t)ceil_div(kv, P);
    const int32_t* pl = pages + p->page_indptr_copy[r];
    for (int32_t i = 0; i + 1 < need; ++i) {
      const int32_t old = seen[pl[i]];
      slots += P - old;
      seen[pl[i]] = (uint8_t)P;
    }
    if (need > 0) {
      const int32_t last = kv - (need - 1) * P;
      const int32_t old = seen[pl[need - 1]];
      const int32_t nv = std::max(old, last);
      slots += nv - old;
      seen[pl[need - 1]] = (uint8_t)nv;
    }
  }
  return slots * p->tok_bytes;
}
}  // namespace

extern "C" pps_status pps_plan_get_info(const pps_plan* p, pps_plan_info* info) {
  if (!p || !info) return PPS_ERR_INVALID_ARGUMENT;
  if (p->kv_bytes_unique < 0) {
    try {
      p->kv_bytes_unique = unique_kv_bytes(p);
    } catch (const std::bad_alloc&) {
      return PPS_ERR_NO_MEMORY;
    }
  }
  std::memset(info, 0, sizeof(*info));
  info->num_requests = p->num_requests;
  info->num_tokens = p->num_tokens;
  info->num_q_heads = p->shape.num_q_heads;
  info->num_kv_heads = p->shape.num_kv_heads;
  info->head_dim = p->shape.head_dim;
  info->page_size = p->shape.page_size;
  info->num_groups = p->num_groups;
  info->num_bw_tasks = p->num_bw;
  info->num_mma_tasks = p->num_mma;
  info->num_partials = p->num_partials;
  info->num_merge_tokens = p->num_merge_tokens;
  info->table_bytes = (int64_t)p->table_bytes;
  info->workspace_bytes = (int64_t)p->workspace_bytes;
  info->kv_bytes_unique = p->kv_bytes_unique;
  info->kv_bytes_read = p->kv_bytes_read;
  info->flops_mma = p->flops_mma;
  info->flops_total = p->flops_total;
  info->kv_bytes_bw = p->kv_bytes_bw;
  info->flops_mma_issued = p->flops_mma_issued;
  info->num_tree_requests = p->num_tree_requests;
  info->small_rows_on_tensor = p->shape.small_tt;
  return PPS_OK;
}

extern "C" pps_status pps_plan_get_array(const pps_plan* p, int32_t which, const int32_t** data,
                                         int64_t* count) {
  if (!p || !data || !count) return PPS_ERR_INVALID_ARGUMENT;
  const int32_t* img = p->image.data;
  const auto& L = p->layout;
  switch (which) {
    case PPS_ARRAY_BW_TASKS: *data = img + L.bw_tasks; *count = p->num_bw * PPS_TASK_INTS; break;
    case PPS_ARRAY_MMA_TASKS: *data = img + L.mma_tasks; *count = p->num_mma * PPS_TASK_INTS; break;
    case PPS_ARRAY_ROWS: *data = img + L.rows; *count = p->num_rows; break;
    case PPS_ARRAY_PAGES: *data = img + L.pages; *count = p->num_pages_listed; break;
    case PPS_ARRAY_MERGE_TOKENS: *data = img + L.merge_tokens; *count = p->num_merge_tokens; break;
    case PPS_ARRAY_MERGE_INDPTR: *data = img + L.merge_indptr; *count = p->num_merge_tokens + 1; break;
    case PPS_ARRAY_MERGE_PIDS: *data = img + L.merge_pids; *count = p->num_merge_pids; break;
    case PPS_ARRAY_TREE_MASK:
      *data = img + L.tree_mask;
      *count = p->has_tree ? 2LL * p->num_tokens : 0;
      break;
    case PPS_ARRAY_TT_CTA:
      *data = img + L.tt_cta;
      *count = p->shape.tt_ctas > 0 ? p->shape.tt_ctas + 1 : 0;
      break;
    default: return PPS_ERR_INVALID_ARGUMENT;
  }
  return PPS_OK;
}

// Batch partition over GPUs (pps_partition): radix subtrees whole, greedy by
// work, largest first.  Rules in pps.h.
extern "C" pps_status pps_partition(const int32_t* q_indptr, const int32_t* kv_len,
                                    const int32_t* page_indptr, const int32_t* page_indices,
                                    int32_t num_requests, int32_t page_size, int32_t num_parts,
                                    int32_t* out_part, int64_t* out_load) {
  if (num_requests < 0 || num_parts <= 0 || page_size <= 0 || !out_part ||
      (num_requests > 0 && (!q_indptr || !kv_len || !page_indptr)))
    return PPS_ERR_INVALID_ARGUMENT;
  try {
    const int32_t R = num_requests;
    struct Sub {
      int64_t work = 0;
      int32_t first_req = 0;
      std::vector<int32_t> members;
    };
    std::vector<Sub> subs;
    std::unordered_map<int32_t, int32_t> by_page;          // first cached page -> subtree
    for (int32_t r = 0; r < R; ++r) {
      const int32_t q = q_indptr[r + 1] - q_indptr[r];
      if (q < 0 || kv_len[r] < q) return PPS_ERR_INVALID_ARGUMENT;
      const int32_t cached = kv_len[r] - q;
      int32_t id = -1;
      if (cached >= page_size) {
        if (!page_indices || page_indptr[r + 1] <= page_indptr[r]) return PPS_ERR_PAGE_TABLE;
        const int32_t pg = page_indices[page_indptr[r]];
        auto it = by_page.find(pg);
        if (it != by_page.end()) id = it->second;
        else by_page.emplace(pg, id = (int32_t)subs.size());
      }
      if (id < 0 || id == (int32_t)subs.size()) {
        id = (int32_t)subs.size();
        subs.emplace_back();
        subs.back().first_req = r;
      }
      subs[id].work += (int64_t)std::max(1, q) * kv_len[r];
      subs[id].members.push_back(r);
    }
    std::vector<int32_t> order(subs.size());
    std::iota(order.begin(), order.end(), 0);
    std::sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
      if (subs[a].work != subs[b].work) return subs[a].work > subs[b].work;
      return subs[a].first_req < subs[b].first_req;
    });
    std::vector<int64_t> load((size_t)num_parts, 0);
    for (int32_t k : order) {
      int32_t best = 0;
      for (int32_t p = 1; p < num_parts; ++p)
        if (load[p] < load[best]) best = p;
      load[best] += subs[k].work;
      for (int32_t r : subs[k].members) out_part[r] = best;
    }
    if (out_load)
      for (int32_t p = 0; p < num_parts; ++p) out_load[p] = load[p];
  } catch (const std::bad_alloc&) {
    return PPS_ERR_NO_MEMORY;
  }
  return PPS_OK;
}
