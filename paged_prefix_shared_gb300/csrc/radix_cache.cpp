// Host radix-tree prefix cache with a page allocator (pps_cache_*): produces the
// per-request page lists that pps_kv_append and pps_attn_plan consume.
//
// SGLang review (pith.science/p/2312.07104), "Core claim": RadixAttention keeps
// finished requests' KV in a radix tree for reuse by later requests sharing a
// prefix.  XY-Serve review (pith.science/paper/ABCKJ6RF), "Assumptions & free
// parameters" and Fig. 7: PagedAttention block table plus radix tree under
// copy-on-write and eviction, with token-wise reuse.  The rules (one node per
// page, greedy longest match capped at n - 1 tokens, copy-on-write of a partly
// matched page, lowest free page first, LRU or LFU eviction of unpinned leaves,
// duplicate pages dropped on insertion) are spelled out in pps.h.
//
// Layout: nodes live in a slot vector (slots reused after eviction); each
// node's chunk is P ints in one flat vector.  Children are found through a hash
// map keyed by (parent, first token), so matching touches only children that
// share the next token.  Evictable leaves sit in an ordered set keyed by the
// policy's order, updated whenever a node's use, hits, children or page holders
// change.
#include <algorithm>
#include <cstring>
#include <new>
#include <set>
#include <tuple>
#include <unordered_map>
#include <vector>

#include "pps.h"

namespace {

struct Node {
  int32_t page = -1;
  int32_t parent = -1;       // node slot, -1 = root
  int32_t len = 0;           // tokens in the chunk (1..P)
  int64_t last = 0;
  int64_t hits = 0;
  int32_t nchild = 0;
  bool alive = false;
  bool in_ev = false;
  std::tuple<int64_t, int64_t, int32_t, int32_t> ev_key{};
};

struct Request {
  std::vector<int32_t> tokens, pages, path;
};

}  // namespace

struct pps_cache {
  int32_t P = 0, num_pages = 0, policy = PPS_CACHE_LRU;
  int64_t tick = 0;
  std::vector<int32_t> holders;      // per page
  std::vector<int32_t> page_node;    // per page: tree node slot holding it, or -1
  std::set<int32_t> free_pages;
  std::vector<Node> nodes;
  std::vector<int32_t> chunk;        // nodes.size() * P
  std::vector<int32_t> free_slots;
  std::unordered_map<uint64_t, std::vector<int32_t>> kids;   // (parent, first token) -> slots
  std::set<std::tuple<int64_t, int64_t, int32_t, int32_t>> evictable;
  std::unordered_map<int32_t, Request> requests;
  int32_t next_request = 0;
  int64_t evictions = 0, reused_tokens = 0, begun_tokens = 0, live_nodes = 0;

  static uint64_t kid_key(int32_t parent, int32_t first) {
    return ((uint64_t)(uint32_t)(parent + 1) << 32) | (uint32_t)first;
  }
  const int32_t* chunk_of(int32_t s) const { return chunk.data() + (size_t)s * P; }

  void update_ev(int32_t s) {
    Node& n = nodes[s];
    const bool should = n.alive && n.nchild == 0 && holders[n.page] == 1;
    std::tuple<int64_t, int64_t, int32_t, int32_t> key =
        policy == PPS_CACHE_LRU ? std::make_tuple(n.last, (int64_t)0, n.page, s)
                                : std::make_tuple(n.hits, n.last, n.page, s);
    if (n.in_ev && (!should || key != n.ev_key)) {
      evictable.erase(n.ev_key);
      n.in_ev = false;
    }
    if (should && !n.in_ev) {
      evictable.insert(key);
      n.ev_key = key;
      n.in_ev = true;
    }
  }
  void hold(int32_t p) {
    if (holders[p]++ == 0) free_pages.erase(p);
    if (page_node[p] >= 0) update_ev(page_node[p]);
  }
  void release(int32_t p) {
    if (--holders[p] == 0) free_pages.insert(p);
    if (page_node[p] >= 0) update_ev(page_node[p]);
  }
  void touch(int32_t s, bool hit) {
    nodes[s].last = tick;
    if (hit) ++nodes[s].hits;
    update_ev(s);
  }
  void evict_one() {
    const int32_t s = std::get<3>(*evictable.begin());
    Node& n = nodes[s];
    evictable.erase(evictable.begin());
    n.in_ev = false;
    auto it = kids.find(kid_key(n.parent, chunk_of(s)[0]));
    auto& v = it->second;
    v.erase(std::find(v.begin(), v.end(), s));
    if (v.empty()) kids.erase(it);
    const int32_t page = n.page, parent = n.parent;
    n.alive = false;
    page_node[page] = -1;
    free_slots.push_back(s);
    --live_nodes;
    ++evictions;
    release(page);
    if (parent >= 0) {
      --nodes[parent].nchild;
      update_ev(parent);
    }
  }
  // Takes `count` pages (lowest free id first, evicting as needed).  On
  // failure gives back what it took and returns false.
  bool allocate(int64_t count, std::vector<int32_t>& out) {
    const size_t base = out.size();
    for (int64_t k = 0; k < count; ++k) {
      if (free_pages.empty()) {
        if (evictable.empty()) {
          for (size_t j = base; j < out.size(); ++j) release(out[j]);
          out.resize(base);
          return false;
        }
        evict_one();
      }
      const int32_t p = *free_pages.begin();
      hold(p);
      out.push_back(p);
    }
    return true;
  }
  int32_t new_node(int32_t parent, int32_t page, const int32_t* toks, int32_t len) {
    int32_t s;
    if (!free_slots.empty()) {
      s = free_slots.back();
      free_slots.pop_back();
    } else {
      s = (int32_t)nodes.size();
      nodes.emplace_back();
      chunk.resize(chunk.size() + P);
    }
    Node& n = nodes[s];
    n = Node{};
    n.page = page;
    n.parent = parent;
    n.len = len;
    n.last = tick;
    n.alive = true;
    std::memcpy(chunk.data() + (size_t)s * P, toks, (size_t)len * 4);
    kids[kid_key(parent, toks[0])].push_back(s);
    page_node[page] = s;
    ++live_nodes;
    if (parent >= 0) {
      ++nodes[parent].nchild;
      update_ev(parent);
    }
    update_ev(s);
    return s;
  }
};

extern "C" pps_status pps_cache_create(int32_t num_pages, int32_t page_size, int32_t policy,
                                       pps_cache** out) {
  if (!out) return PPS_ERR_INVALID_ARGUMENT;
  *out = nullptr;
  if (num_pages <= 0 || page_size <= 0 || (policy != PPS_CACHE_LRU && policy != PPS_CACHE_LFU))
    return PPS_ERR_INVALID_ARGUMENT;
  pps_cache* c = new (std::nothrow) pps_cache;
  if (!c) return PPS_ERR_NO_MEMORY;
  try {
    c->P = page_size;
    c->num_pages = num_pages;
    c->policy = policy;
    c->holders.assign((size_t)num_pages, 0);
    c->page_node.assign((size_t)num_pages, -1);
    for (int32_t p = 0; p < num_pages; ++p) c->free_pages.insert(c->free_pages.end(), p);
  } catch (const std::bad_alloc&) {
    delete c;
    return PPS_ERR_NO_MEMORY;
  }
  *out = c;
  return PPS_OK;
}

extern "C" pps_status pps_cache_destroy(pps_cache* c) {
  delete c;
  return PPS_OK;
}

extern "C" pps_status pps_cache_begin(pps_cache* c, const int32_t* tokens, int32_t n,
                                      int32_t* out_request, int32_t* out_cached_len,
                                      int32_t* out_copy) {
  if (!c || !tokens || n <= 0 || !out_request || !out_cached_len || !out_copy)
    return PPS_ERR_INVALID_ARGUMENT;
  try {
    ++c->tick;
    const int32_t P = c->P, limit = n - 1;
    int32_t node = -1, i = 0, partial = -1, partial_l = 0;
    std::vector<int32_t> path;
    while (i < n) {
      int32_t best = -1, best_l = 0;
      auto it = c->kids.find(pps_cache::kid_key(node, tokens[i]));
      if (it != c->kids.end()) {
        for (int32_t ch : it->second) {
          const Node& nd = c->nodes[ch];
          const int32_t* ck = c->chunk_of(ch);
          const int32_t m = std::min(nd.len, n - i);
          int32_t l = 0;
          while (l < m && ck[l] == tokens[i + l]) ++l;
          l = std::min(l, std::max(0, limit - i));
          if (l > best_l || (l == best_l && l > 0 && nd.page < c->nodes[best].page)) {
            best = ch;
            best_l = l;
          }
        }
      }
      if (best < 0) break;
      if (best_l == P) {
        path.push_back(best);
        node = best;
        i += P;
        continue;
      }
      partial = best;
      partial_l = best_l;
      break;
    }
    for (int32_t s : path) {
      c->hold(c->nodes[s].page);
      c->touch(s, true);
    }
    int32_t src = -1;
    if (partial >= 0) {
      c->touch(partial, true);
      src = c->nodes[partial].page;
      c->hold(src);                       // kept while pages are taken
    }
    Request req;
    req.pages.reserve((size_t)(n + P - 1) / P);
    for (int32_t s : path) req.pages.push_back(c->nodes[s].page);
    const int64_t need = (int64_t)(n + P - 1) / P - (int64_t)path.size();
    if (!c->allocate(need, req.pages)) {
      for (int32_t s : path) c->release(c->nodes[s].page);
      if (src >= 0) c->release(src);
      return PPS_ERR_CACHE_FULL;
    }
    int32_t cached = i;
    out_copy[0] = out_copy[1] = -1;
    out_copy[2] = 0;
    if (partial >= 0) {
      c->release(src);
      out_copy[0] = src;
      out_copy[1] = req.pages[path.size()];
      out_copy[2] = partial_l;
      cached += partial_l;
    }
    req.tokens.assign(tokens, tokens + n);
    req.path = std::move(path);
    const int32_t rid = c->next_request++;
    c->requests.emplace(rid, std::move(req));
    c->reused_tokens += cached;
    c->begun_tokens += n;
    *out_request = rid;
    *out_cached_len = cached;
  } catch (const std::bad_alloc&) {
    return PPS_ERR_NO_MEMORY;
  }
  return PPS_OK;
}

extern "C" pps_status pps_cache_extend(pps_cache* c, int32_t request, const int32_t* tokens,
                                       int32_t m, int32_t* out_first_position) {
  if (!c || m < 0 || (m > 0 && !tokens)) return PPS_ERR_INVALID_ARGUMENT;
  auto it = c->requests.find(request);
  if (it == c->requests.end()) return PPS_ERR_INVALID_ARGUMENT;
  try {
    ++c->tick;
    Request& r = it->second;
    const int64_t n0 = (int64_t)r.tokens.size(), n1 = n0 + m;
    const int64_t need = (n1 + c->P - 1) / c->P - (int64_t)r.pages.size();
    if (need > 0 && !c->allocate(need, r.pages)) return PPS_ERR_CACHE_FULL;
    r.tokens.insert(r.tokens.end(), tokens, tokens + m);
    if (out_first_position) *out_first_position = (int32_t)n0;
  } catch (const std::bad_alloc&) {
    return PPS_ERR_NO_MEMORY;
  }
  return PPS_OK;
}

extern "C" pps_status pps_cache_finish(pps_cache* c, int32_t request, int32_t insert) {
  if (!c) return PPS_ERR_INVALID_ARGUMENT;
  auto it = c->requests.find(request);
  if (it == c->requests.end()) return PPS_ERR_INVALID_ARGUMENT;
  try {
    ++c->tick;
    Request r = std::move(it->second);
    c->requests.erase(it);
    const int32_t P = c->P;
    const int64_t n = (int64_t)r.tokens.size();
    size_t k = r.path.size();
    if (insert) {
      int32_t node = -1;
      for (int32_t s : r.path) {
        c->touch(s, false);
        node = s;
      }
      while ((int64_t)k * P < n) {
        const int32_t* ck = r.tokens.data() + k * P;
        const int32_t len = (int32_t)std::min<int64_t>(P, n - (int64_t)k * P);
        const int32_t page = r.pages[k];
        int32_t same = -1;
        auto f = c->kids.find(pps_cache::kid_key(node, ck[0]));
        if (f != c->kids.end())
          for (int32_t ch : f->second)
            if (c->nodes[ch].len == len && std::memcmp(c->chunk_of(ch), ck, (size_t)len * 4) == 0 &&
                (same < 0 || c->nodes[ch].page < c->nodes[same].page))
              same = ch;
        int32_t next;
        if (same >= 0) {
          c->release(page);
          c->touch(same, false);
          next = same;
        } else {
          next = c->new_node(node, page, ck, len);
        }
        node = next;
        ++k;
        if (len < P) break;
      }
    }
    for (size_t j = k; j < r.pages.size(); ++j) c->release(r.pages[j]);
    for (int32_t s : r.path) c->release(c->nodes[s].page);
  } catch (const std::bad_alloc&) {
    return PPS_ERR_NO_MEMORY;
  }
  return PPS_OK;
}

extern "C" pps_status pps_cache_request_pages(const pps_cache* c, int32_t request,
                                              const int32_t** pages, int32_t* num_pages,
                                              int32_t* num_tokens) {
  if (!c || !pages || !num_pages || !num_tokens) return PPS_ERR_INVALID_ARGUMENT;
  auto it = c->requests.find(request);
  if (it == c->requests.end()) return PPS_ERR_INVALID_ARGUMENT;
  *pages = it->second.pages.data();
  *num_pages = (int32_t)it->second.pages.size();
  *num_tokens = (int32_t)it->second.tokens.size();
  return PPS_OK;
}

extern "C" pps_status pps_cache_get_stats(const pps_cache* c, pps_cache_stats* s) {
  if (!c || !s) return PPS_ERR_INVALID_ARGUMENT;
  std::memset(s, 0, sizeof(*s));
  s->num_pages = c->num_pages;
  s->page_size = c->P;
  s->free_pages = (int32_t)c->free_pages.size();
  s->active_requests = (int32_t)c->requests.size();
  s->tree_nodes = c->live_nodes;
  s->evictions = c->evictions;
  s->reused_tokens = c->reused_tokens;
  s->begun_tokens = c->begun_tokens;
  s->tick = c->tick;
  return PPS_OK;
}

extern "C" pps_status pps_cache_dump(const pps_cache* c, int64_t* out, int64_t capacity,
                                     int64_t* needed) {
  if (!c || !needed || capacity < 0 || (capacity > 0 && !out)) return PPS_ERR_INVALID_ARGUMENT;
  const int64_t rec = 5 + c->P;
  *needed = c->live_nodes * rec;
  if (capacity < *needed) return capacity == 0 ? PPS_OK : PPS_ERR_INVALID_ARGUMENT;
  int64_t o = 0;
  for (size_t s = 0; s < c->nodes.size(); ++s) {
    const Node& n = c->nodes[s];
    if (!n.alive) continue;
    out[o++] = n.page;
    out[o++] = n.parent >= 0 ? c->nodes[n.parent].page : -1;
    out[o++] = n.len;
    out[o++] = n.last;
    out[o++] = n.hits;
    for (int32_t j = 0; j < c->P; ++j) out[o++] = j < n.len ? c->chunk_of((int32_t)s)[j] : -1;
  }
  return PPS_OK;
}

extern "C" pps_status pps_cache_extend_batch(pps_cache* c, const int32_t* requests,
                                             const int32_t* token_indptr, const int32_t* tokens,
                                             int32_t count, int32_t* out_first_positions,
                                             int32_t* out_done) {
  if (!c || count < 0 || (count > 0 && (!requests || !token_indptr || !tokens)) || !out_done)
    return PPS_ERR_INVALID_ARGUMENT;
  *out_done = 0;
  for (int32_t i = 0; i < count; ++i) {
    const int32_t m = token_indptr[i + 1] - token_indptr[i];
    if (m < 0) return PPS_ERR_INVALID_ARGUMENT;
    int32_t first = 0;
    const pps_status st = pps_cache_extend(c, requests[i], tokens + token_indptr[i], m, &first);
    if (st != PPS_OK) return st;
    if (out_first_positions) out_first_positions[i] = first;
    *out_done = i + 1;
  }
  return PPS_OK;
}

extern "C" pps_status pps_cache_tables(const pps_cache* c, const int32_t* requests, int32_t count,
                                       int32_t* kv_len, int32_t* page_indptr,
                                       int32_t* page_indices, int64_t capacity) {
  if (!c || count < 0 || !page_indptr || (count > 0 && (!requests || !kv_len)))
    return PPS_ERR_INVALID_ARGUMENT;
  int64_t off = 0;
  page_indptr[0] = 0;
  for (int32_t i = 0; i < count; ++i) {
    auto it = c->requests.find(requests[i]);
    if (it == c->requests.end()) return PPS_ERR_INVALID_ARGUMENT;
    const auto& pg = it->second.pages;
    if (off + (int64_t)pg.size() > capacity || (!page_indices && !pg.empty()))
      return PPS_ERR_INVALID_ARGUMENT;
    if (!pg.empty()) std::memcpy(page_indices + off, pg.data(), pg.size() * 4);
    off += (int64_t)pg.size();
    if (off > INT32_MAX) return PPS_ERR_INVALID_ARGUMENT;
    page_indptr[i + 1] = (int32_t)off;
    kv_len[i] = (int32_t)it->second.tokens.size();
  }
  return PPS_OK;
}
