// Host token-wise budget scheduler (pps_sched_*): forms each step's mixed
// batch from the prefill, decode and verify queues.
//
// XY-Serve review (pith.science/paper/ABCKJ6RF), "Core claim": a token-wise
// scheduler selects a budgeted chunk of tokens from mixed prefill, decode and
// verify queues (SplitFuse-style chunking); Fig. 6: prefills are split so every
// scheduled chunk stays within the budget, and some slots are reserved for
// decode and speculative tokens.  The rules are spelled out in pps.h.
//
// Generation requests sit in a list in the order they started generating,
// prefill requests in arrival order; a hash map from request id to list
// position makes removal O(1).  A step walks the generation list once and the
// prefill list until the budget or the prefill room runs out.
#include <algorithm>
#include <iterator>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "pps.h"

namespace {
struct Entry {
  int32_t request;
  int32_t remaining;    // prompt tokens still to schedule (prefill list only)
  int32_t gen_tokens;   // tokens per generation step
};
}  // namespace

struct pps_sched {
  int32_t budget = 0, reserved = 0;
  std::list<Entry> gen, prefill;
  std::unordered_map<int32_t, std::pair<bool, std::list<Entry>::iterator>> where;  // (in prefill?, pos)
};

extern "C" pps_status pps_sched_create(int32_t budget, int32_t reserved, pps_sched** out) {
  if (!out) return PPS_ERR_INVALID_ARGUMENT;
  *out = nullptr;
  if (budget <= 0 || reserved < 0 || reserved > budget) return PPS_ERR_INVALID_ARGUMENT;
  pps_sched* s = new (std::nothrow) pps_sched;
  if (!s) return PPS_ERR_NO_MEMORY;
  s->budget = budget;
  s->reserved = reserved;
  *out = s;
  return PPS_OK;
}

extern "C" pps_status pps_sched_destroy(pps_sched* s) {
  delete s;
  return PPS_OK;
}

extern "C" pps_status pps_sched_add(pps_sched* s, int32_t request, int32_t prompt_tokens,
                                    int32_t gen_tokens) {
  if (!s || prompt_tokens < 0 || gen_tokens <= 0 || s->where.count(request))
    return PPS_ERR_INVALID_ARGUMENT;
  try {
    if (prompt_tokens == 0) {
      s->gen.push_back({request, 0, gen_tokens});
      s->where[request] = {false, std::prev(s->gen.end())};
    } else {
      s->prefill.push_back({request, prompt_tokens, gen_tokens});
      s->where[request] = {true, std::prev(s->prefill.end())};
    }
  } catch (const std::bad_alloc&) {
    return PPS_ERR_NO_MEMORY;
  }
  return PPS_OK;
}

extern "C" pps_status pps_sched_remove(pps_sched* s, int32_t request) {
  if (!s) return PPS_ERR_INVALID_ARGUMENT;
  auto it = s->where.find(request);
  if (it == s->where.end()) return PPS_ERR_INVALID_ARGUMENT;
  (it->second.first ? s->prefill : s->gen).erase(it->second.second);
  s->where.erase(it);
  return PPS_OK;
}

extern "C" pps_status pps_sched_set_gen_tokens(pps_sched* s, int32_t request, int32_t gen_tokens) {
  if (!s || gen_tokens <= 0) return PPS_ERR_INVALID_ARGUMENT;
  auto it = s->where.find(request);
  if (it == s->where.end()) return PPS_ERR_INVALID_ARGUMENT;
  it->second.second->gen_tokens = gen_tokens;
  return PPS_OK;
}

extern "C" pps_status pps_sched_step(pps_sched* s, int32_t* out_requests, int32_t* out_tokens,
                                     int32_t* out_is_prefill, int32_t capacity,
                                     int32_t* out_count) {
  if (!s || !out_count || capacity < 0 ||
      (capacity > 0 && (!out_requests || !out_tokens || !out_is_prefill)))
    return PPS_ERR_INVALID_ARGUMENT;
  *out_count = 0;
  // Decide first, apply once the output fits.
  int32_t left = s->budget, room = s->budget - s->reserved, n = 0;
  for (const Entry& e : s->gen)
    if (e.gen_tokens <= left) {
      left -= e.gen_tokens;
      ++n;
    }
  std::vector<std::pair<std::list<Entry>::iterator, int32_t>> takes;
  for (auto it = s->prefill.begin(); it != s->prefill.end(); ++it) {
    const int32_t take = std::min(it->remaining, std::min(room, left));
    if (take <= 0) break;
    takes.push_back({it, take});
    left -= take;
    room -= take;
  }
  n += (int32_t)takes.size();
  if (n > capacity) return PPS_ERR_INVALID_ARGUMENT;
  int32_t k = 0;
  left = s->budget;
  for (const Entry& e : s->gen)
    if (e.gen_tokens <= left) {
      left -= e.gen_tokens;
      out_requests[k] = e.request;
      out_tokens[k] = e.gen_tokens;
      out_is_prefill[k] = 0;
      ++k;
    }
  for (auto& t : takes) {
    out_requests[k] = t.first->request;
    out_tokens[k] = t.second;
    out_is_prefill[k] = 1;
    ++k;
    t.first->remaining -= t.second;
  }
  // prompts done this step start generating at the end of the list
  for (auto& t : takes) {
    if (t.first->remaining != 0) continue;
    const Entry e = *t.first;
    s->prefill.erase(t.first);
    s->gen.push_back(e);
    s->where[e.request] = {false, std::prev(s->gen.end())};
  }
  *out_count = k;
  return PPS_OK;
}

extern "C" pps_status pps_sched_counts(const pps_sched* s, int32_t* prefill_requests,
                                       int64_t* prefill_tokens, int32_t* gen_requests) {
  if (!s || !prefill_requests || !prefill_tokens || !gen_requests) return PPS_ERR_INVALID_ARGUMENT;
  *prefill_requests = (int32_t)s->prefill.size();
  int64_t t = 0;
  for (const Entry& e : s->prefill) t += e.remaining;
  *prefill_tokens = t;
  *gen_requests = (int32_t)s->gen.size();
  return PPS_OK;
}
