"""Reference radix-tree prefix cache with a page allocator (test infrastructure only).

Plain and slow on purpose: the tree is a flat dict of nodes, every lookup scans
all nodes, nothing is indexed.  It defines, step by step, what the library's
host cache must do; tests compare the two operation by operation.

Sources (page title and section):
* SGLang review, "SGLang: Efficient Execution of Structured Language Model
  Programs" (pith.science/p/2312.07104), "Core claim": RadixAttention keeps
  the KV cache of finished requests in a radix tree so later requests that
  share a prefix reuse it.
* XY-Serve review, "Tackling the Dynamicity in a Production LLM Serving
  System ..." (pith.science/paper/ABCKJ6RF), "Assumptions & free
  parameters": a PagedAttention block table plus a radix tree keeps K/V
  semantics under copy-on-write and eviction; Fig. 7, token-wise K/V cache
  reuse (a prefix is reused down to the token, not only whole pages).
* attentionhub.org listing, the cache-replacement entries: recency (LRU)
  and frequency (LFU) eviction.

Rules (the pages fix none of them; these are the plainest that satisfy the
sources, and the library follows the same ones):
* One tree node = one page: a chunk of up to P token ids.  A chunk of fewer
  than P tokens (a request's partly filled last page) is always a leaf.
* Matching (``begin``) walks from the root.  Among the children, the one whose
  chunk shares the longest prefix with the next tokens wins (ties: lowest
  page id).  A whole full page matched descends; otherwise, if the shared
  prefix is non-empty, it is reused token-wise: copy-on-write of those slots
  into the request's first new page.  At most n - 1 tokens are reused, so
  every request computes at least its last token.
* Pages are handed out lowest id first.  With no free page, one evictable
  node is evicted (its page freed) and allocation retries.  Evictable: a leaf
  whose page no active request holds.  Victim: smallest (last use, page) for
  LRU, smallest (hits, last use, page) for LFU.  If nothing is evictable the
  call fails with CacheFull after giving back the pages it took (evictions
  already done stay done).
* Every call advances a tick.  A node's last use is the tick of the last call
  that matched, copied from or walked it; its hits count the ``begin`` calls
  that reused it (fully or token-wise).
* ``finish`` inserts the request's pages below its matched path: a chunk equal
  to an existing child's chunk drops the request's page (freed if nobody else
  holds it) and walks into that child; otherwise the page becomes a new node
  (last use = now, hits = 0).  Insertion stops after a partial chunk.
  ``finish(insert=False)`` only releases the request.
* A page is held by each tree node on it and by each active request listing
  it; it is free when nobody holds it.
"""
from __future__ import annotations


class CacheFull(Exception):
    """No free page and nothing evictable."""


def _lcp(a, b):
    n = 0
    for x, y in zip(a, b):
        if x != y:
            break
        n += 1
    return n


class RadixCacheOracle:
    def __init__(self, num_pages, page_size, policy="lru"):
        if policy not in ("lru", "lfu"):
            raise ValueError(policy)
        self.P = int(page_size)
        self.num_pages = int(num_pages)
        self.policy = policy
        self.holders = [0] * self.num_pages
        self.nodes = {}            # id -> {"page", "chunk", "parent", "last", "hits"}
        self.next_node = 0
        self.tick = 0
        self.requests = {}         # id -> {"tokens", "pages", "path"}
        self.next_request = 0
        self.evictions = []        # pages of evicted nodes, in order
        self.reused_tokens = 0
        self.begun_tokens = 0

    # ---- helpers -------------------------------------------------------------
    def _children(self, parent):
        return [i for i, n in self.nodes.items() if n["parent"] == parent]

    def _touch(self, node):
        self.nodes[node]["last"] = self.tick

    def _evictable(self):
        out = []
        for i, n in self.nodes.items():
            if self._children(i):
                continue
            if self.holders[n["page"]] == 1:      # the node's own hold only
                out.append(i)
        return out

    def _victim_key(self, i):
        n = self.nodes[i]
        if self.policy == "lru":
            return (n["last"], n["page"])
        return (n["hits"], n["last"], n["page"])

    def _allocate(self, count):
        taken = []
        for _ in range(count):
            free = [p for p in range(self.num_pages) if self.holders[p] == 0]
            if not free:
                cand = self._evictable()
                if not cand:
                    for p in taken:
                        self.holders[p] -= 1
                    raise CacheFull()
                v = min(cand, key=self._victim_key)
                page = self.nodes[v]["page"]
                del self.nodes[v]
                self.holders[page] -= 1
                self.evictions.append(page)
                free = [p for p in range(self.num_pages) if self.holders[p] == 0]
            p = min(free)
            self.holders[p] += 1
            taken.append(p)
        return taken

    # ---- operations ----------------------------------------------------------
    def begin(self, tokens):
        """Start a request.  Returns (request id, cached_len, copy) where
        copy is None or (src_page, dst_page, slots)."""
        self.tick += 1
        tokens = [int(t) for t in tokens]
        n = len(tokens)
        if n == 0:
            raise ValueError("empty request")
        P = self.P
        limit = n - 1
        node, i, path, partial = -1, 0, [], None
        while True:
            best, best_l = None, 0
            for c in self._children(node):
                chunk = self.nodes[c]["chunk"]
                l = min(_lcp(chunk, tokens[i:i + len(chunk)]), max(0, limit - i))
                if l > best_l or (l == best_l and l > 0 and
                                  self.nodes[c]["page"] < self.nodes[best]["page"]):
                    best, best_l = c, l
            if best is None:
                break
            if best_l == P:
                path.append(best)
                node = best
                i += P
                continue
            partial = (best, best_l)
            break
        for c in path:
            self.holders[self.nodes[c]["page"]] += 1
            self._touch(c)
            self.nodes[c]["hits"] += 1
        src = None
        if partial is not None:
            c, l = partial
            self._touch(c)
            self.nodes[c]["hits"] += 1
            src = self.nodes[c]["page"]
            self.holders[src] += 1                  # kept while pages are taken
        need = -(-n // P) - len(path)
        try:
            pages = self._allocate(need)
        except CacheFull:
            for c in path:
                self.holders[self.nodes[c]["page"]] -= 1
            if src is not None:
                self.holders[src] -= 1
            raise
        copy = None
        cached = i
        if partial is not None:
            self.holders[src] -= 1
            copy = (src, pages[0], partial[1])
            cached += partial[1]
        rid = self.next_request
        self.next_request += 1
        self.requests[rid] = {"tokens": tokens,
                              "pages": [self.nodes[c]["page"] for c in path] + pages,
                              "path": path}
        self.reused_tokens += cached
        self.begun_tokens += n
        return rid, cached, copy

    def extend(self, rid, tokens):
        """Append tokens to an active request (decode).  Returns the number of
        tokens it held before (the first new position)."""
        self.tick += 1
        req = self.requests[rid]
        n0 = len(req["tokens"])
        n1 = n0 + len(tokens)
        need = -(-n1 // self.P) - len(req["pages"])
        if need > 0:
            req["pages"] += self._allocate(need)
        req["tokens"] += [int(t) for t in tokens]
        return n0

    def finish(self, rid, insert=True):
        self.tick += 1
        req = self.requests.pop(rid)
        P = self.P
        if insert:
            node = -1
            for c in req["path"]:
                self._touch(c)
                node = c
            k = len(req["path"])
            n = len(req["tokens"])
            while k * P < n:
                chunk = tuple(req["tokens"][k * P:(k + 1) * P])
                page = req["pages"][k]
                same = [c for c in self._children(node) if self.nodes[c]["chunk"] == chunk]
                if same:
                    c = min(same, key=lambda x: self.nodes[x]["page"])
                    self.holders[page] -= 1
                    self._touch(c)
                else:
                    c = self.next_node
                    self.next_node += 1
                    self.nodes[c] = {"page": page, "chunk": chunk, "parent": node,
                                     "last": self.tick, "hits": 0}
                node = c
                k += 1
                if len(chunk) < P:
                    break
            for page in req["pages"][k:]:          # pages past the tokens (none expected)
                self.holders[page] -= 1
        else:
            for page in req["pages"][len(req["path"]):]:
                self.holders[page] -= 1
        for c in req["path"]:
            self.holders[self.nodes[c]["page"]] -= 1

    # ---- views ---------------------------------------------------------------
    def pages(self, rid):
        return list(self.requests[rid]["pages"])

    def num_free(self):
        return sum(1 for h in self.holders if h == 0)

    def node_sequences(self):
        """Token sequence (root to node) of every tree node, with its page."""
        out = []
        for i in self.nodes:
            seq, n = [], i
            while n != -1:
                seq = list(self.nodes[n]["chunk"]) + seq
                n = self.nodes[n]["parent"]
            out.append((seq, self.nodes[i]["page"]))
        return out
