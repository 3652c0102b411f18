// Serving-step runtime (pps_engine_*): a prefix cache and a token-wise
// scheduler kept together, so one step of a serving loop is two native calls:
// pps_engine_schedule picks the batch (pps_sched_step), pps_engine_commit
// takes the new token ids of its generation entries, extends the cache, moves
// the prefill entries forward and writes the batch's tables for pps_kv_append
// and pps_attn_plan.  Admission (pps_engine_add: pps_cache_begin +
// pps_sched_add) and retirement (pps_engine_finish) are separate calls.
//
// Sources: XY-Serve review (pith.science/paper/ABCKJ6RF), "Core claim"
// (token-wise scheduler over mixed prefill/decode/verify queues, prefix
// caching) and Fig. 6; SGLang review (pith.science/p/2312.07104), "Core claim"
// (radix-tree KV reuse).
#include <algorithm>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pps.h"

namespace {
struct EngReq {
  int32_t prompt_len = 0;     // tokens given to pps_engine_add
  int32_t cached0 = 0;        // of them already cached at admission
  int32_t prefill_done = 0;   // prompt tokens scheduled since
};
}  // namespace

struct pps_engine {
  int32_t page_size = 0;
  pps_cache* cache = nullptr;
  pps_sched* sched = nullptr;
  std::unordered_map<int32_t, EngReq> reqs;
  std::vector<int32_t> b_req, b_tok, b_pre;   // the batch picked by the last schedule call
  bool pending = false;
};

extern "C" pps_status pps_engine_create(int32_t num_pages, int32_t page_size, int32_t policy,
                                        int32_t budget, int32_t reserved, pps_engine** out) {
  if (!out) return PPS_ERR_INVALID_ARGUMENT;
  *out = nullptr;
  pps_engine* e = new (std::nothrow) pps_engine;
  if (!e) return PPS_ERR_NO_MEMORY;
  e->page_size = page_size;
  pps_status st = pps_cache_create(num_pages, page_size, policy, &e->cache);
  if (st == PPS_OK) st = pps_sched_create(budget, reserved, &e->sched);
  if (st != PPS_OK) {
    pps_cache_destroy(e->cache);
    delete e;
    return st;
  }
  *out = e;
  return PPS_OK;
}

extern "C" pps_status pps_engine_destroy(pps_engine* e) {
  if (!e) return PPS_OK;
  pps_sched_destroy(e->sched);
  pps_cache_destroy(e->cache);
  delete e;
  return PPS_OK;
}

extern "C" pps_status pps_engine_parts(pps_engine* e, pps_cache** cache, pps_sched** sched) {
  if (!e) return PPS_ERR_INVALID_ARGUMENT;
  if (cache) *cache = e->cache;
  if (sched) *sched = e->sched;
  return PPS_OK;
}

extern "C" pps_status pps_engine_add(pps_engine* e, const int32_t* tokens, int32_t n,
                                     int32_t gen_tokens, int32_t* out_request,
                                     int32_t* out_cached_len, int32_t* out_copy) {
  if (!e || e->pending || gen_tokens <= 0 || !out_request || !out_cached_len || !out_copy)
    return PPS_ERR_INVALID_ARGUMENT;
  pps_status st = pps_cache_begin(e->cache, tokens, n, out_request, out_cached_len, out_copy);
  if (st != PPS_OK) return st;
  st = pps_sched_add(e->sched, *out_request, n - *out_cached_len, gen_tokens);
  if (st != PPS_OK) {
    pps_cache_finish(e->cache, *out_request, 0);
    return st;
  }
  try {
    EngReq r;
    r.prompt_len = n;
    r.cached0 = *out_cached_len;
    e->reqs.emplace(*out_request, r);
  } catch (const std::bad_alloc&) {
    pps_sched_remove(e->sched, *out_request);
    pps_cache_finish(e->cache, *out_request, 0);
    return PPS_ERR_NO_MEMORY;
  }
  return PPS_OK;
}

extern "C" pps_status pps_engine_finish(pps_engine* e, int32_t request, int32_t insert) {
  if (!e || e->pending) return PPS_ERR_INVALID_ARGUMENT;
  auto it = e->reqs.find(request);
  if (it == e->reqs.end()) return PPS_ERR_INVALID_ARGUMENT;
  pps_sched_remove(e->sched, request);
  e->reqs.erase(it);
  return pps_cache_finish(e->cache, request, insert);
}

extern "C" pps_status pps_engine_schedule(pps_engine* e, int32_t* out_requests,
                                          int32_t* out_tokens, int32_t* out_is_prefill,
                                          int32_t capacity, int32_t* out_count) {
  if (!e || e->pending || !out_count) return PPS_ERR_INVALID_ARGUMENT;
  const pps_status st =
      pps_sched_step(e->sched, out_requests, out_tokens, out_is_prefill, capacity, out_count);
  if (st != PPS_OK) return st;
  try {
    e->b_req.assign(out_requests, out_requests + *out_count);
    e->b_tok.assign(out_tokens, out_tokens + *out_count);
    e->b_pre.assign(out_is_prefill, out_is_prefill + *out_count);
  } catch (const std::bad_alloc&) {
    return PPS_ERR_NO_MEMORY;
  }
  e->pending = true;
  return PPS_OK;
}

extern "C" pps_status pps_engine_commit(pps_engine* e, const int32_t* gen_tokens,
                                        int32_t* out_requests, int32_t* q_indptr,
                                        int32_t* cached_len, int32_t* kv_len,
                                        int32_t* page_indptr, int32_t* page_indices,
                                        int64_t page_capacity, int64_t* out_pages_needed,
                                        int32_t* out_count) {
  if (!e || !e->pending || !out_count) return PPS_ERR_INVALID_ARGUMENT;
  const int32_t n = (int32_t)e->b_req.size();
  if (n > 0 && (!out_requests || !q_indptr || !cached_len || !kv_len || !page_indptr ||
                !page_indices))
    return PPS_ERR_INVALID_ARGUMENT;
  *out_count = 0;
  // Room check before anything changes: every entry's pages, plus what the
  // generation entries may add.
  int64_t bound = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t* pages;
    int32_t np, nt;
    if (pps_cache_request_pages(e->cache, e->b_req[i], &pages, &np, &nt) != PPS_OK)
      return PPS_ERR_INVALID_ARGUMENT;
    bound += np + (e->b_pre[i] ? 0 : e->b_tok[i] / e->page_size + 1);
  }
  if (out_pages_needed) *out_pages_needed = bound;
  if (bound > page_capacity) return PPS_ERR_INVALID_ARGUMENT;
  e->pending = false;
  // Generation entries get their tokens appended; one the cache has no page
  // for is left out of this step (the scheduler picks it again next step).
  // Prefill entries move forward (their pages were taken at admission).
  int32_t k = 0;
  int64_t g = 0, off = 0;
  q_indptr[0] = 0;
  page_indptr[0] = 0;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t r = e->b_req[i], t = e->b_tok[i];
    int32_t first;
    if (e->b_pre[i]) {
      EngReq& q = e->reqs[r];
      first = q.cached0 + q.prefill_done;
      q.prefill_done += t;
    } else {
      const pps_status st = pps_cache_extend(e->cache, r, gen_tokens + g, t, &first);
      g += t;
      if (st == PPS_ERR_CACHE_FULL) continue;
      if (st != PPS_OK) return st;
    }
    const int32_t* pages;
    int32_t np, nt;
    pps_cache_request_pages(e->cache, r, &pages, &np, &nt);
    out_requests[k] = r;
    cached_len[k] = first;
    kv_len[k] = first + t;
    q_indptr[k + 1] = q_indptr[k] + t;
    std::memcpy(page_indices + off, pages, (size_t)np * 4);
    off += np;
    page_indptr[k + 1] = (int32_t)off;
    ++k;
  }
  *out_count = k;
  return PPS_OK;
}
