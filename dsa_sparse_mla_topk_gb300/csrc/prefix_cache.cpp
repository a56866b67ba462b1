// KV-only prefix-sharing page allocator (host side).
//
// "Accelerating GLM-5.3-Flash on H200", section 2 "KV-only decode
// RadixCache": requests that share a prefix share its KV pages, so N requests
// with a common prefix of Lp tokens and private suffixes of Ls tokens occupy
// Lp + N·Ls token slots instead of N·(Lp + Ls).  Pages are the unit of
// sharing: a page is shared only when the whole page and everything before it
// match (KV rows depend on the whole causal prefix), so the accounting is
// Lp rounded down to whole pages, plus each request's remaining pages.
//
// The structure is a radix tree with one node per cached page; a node's key
// is the page's token ids and its path from the root is the prefix.  Acquire
// walks the tree page by page, reuses (and references) every matching page,
// takes fresh pages for the rest and inserts the request's full pages so
// later requests can share them; a partial last page stays private.  Release
// drops the references: private pages go back to the free list, cached pages
// stay until the pool runs out, when unreferenced leaves are evicted least
// recently used first.  All calls take one mutex.
#include <stdint.h>

#include <map>
#include <mutex>
#include <new>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

#include "dsa.h"

namespace {

struct Node {
  int32_t page = -1;
  Node* parent = nullptr;
  std::vector<int32_t> tokens;                     // the page's token ids (page_size of them)
  std::unordered_multimap<uint64_t, Node*> kids;   // by hash of the child's tokens
  int32_t refs = 0;
  uint64_t stamp = 0;                              // last acquire or release touching it
};

uint64_t hash_tokens(const int32_t* t, int32_t n) {
  uint64_t h = 1469598103934665603ull;  // FNV-1a over the bytes of the ids
  for (int32_t i = 0; i < n; ++i) {
    uint32_t v = (uint32_t)t[i];
    for (int b = 0; b < 4; ++b) {
      h ^= (v >> (8 * b)) & 0xffu;
      h *= 1099511628211ull;
    }
  }
  return h;
}

}  // namespace

struct dsa_prefix_cache {
  int32_t page_size = 0;
  int32_t num_pages = 0;
  std::mutex mu;
  Node root;
  std::vector<Node*> node_of;     // page id -> its tree node, or null (private or free)
  std::vector<int32_t> priv_refs; // references of private pages
  std::vector<int32_t> free_list;
  std::set<std::pair<uint64_t, int32_t>> evictable;  // (stamp, page) of unreferenced leaves
  uint64_t clock = 0;
  int32_t referenced = 0;         // pages with refs > 0 (tree or private)
  int32_t cached = 0;             // pages in the tree

  bool is_evictable(const Node* n) const { return n != &root && n->refs == 0 && n->kids.empty(); }
  void unmark(Node* n) { evictable.erase({n->stamp, n->page}); }
  void mark_if(Node* n) {
    if (is_evictable(n)) evictable.insert({n->stamp, n->page});
  }

  // one free page, evicting the least recently used unreferenced leaf when needed; -1 if none
  int32_t take_page() {
    if (free_list.empty()) {
      if (evictable.empty()) return -1;
      const int32_t pg = evictable.begin()->second;
      evictable.erase(evictable.begin());
      Node* n = node_of[pg];
      Node* par = n->parent;
      auto range = par->kids.equal_range(hash_tokens(n->tokens.data(), page_size));
      for (auto it = range.first; it != range.second; ++it)
        if (it->second == n) {
          par->kids.erase(it);
          break;
        }
      node_of[pg] = nullptr;
      --cached;
      delete n;
      mark_if(par);  // the parent may now be an unreferenced leaf
      free_list.push_back(pg);
    }
    const int32_t pg = free_list.back();
    free_list.pop_back();
    return pg;
  }

  Node* find_child(Node* n, const int32_t* t) {
    auto range = n->kids.equal_range(hash_tokens(t, page_size));
    for (auto it = range.first; it != range.second; ++it) {
      const std::vector<int32_t>& k = it->second->tokens;
      bool same = true;
      for (int32_t i = 0; i < page_size && same; ++i) same = k[i] == t[i];
      if (same) return it->second;
    }
    return nullptr;
  }

  void ref_node(Node* n) {
    unmark(n);
    if (n->refs++ == 0) ++referenced;
    n->stamp = ++clock;
  }
  void unref_node(Node* n) {
    if (--n->refs == 0) --referenced;
    n->stamp = ++clock;
    mark_if(n);
  }
};

extern "C" {

dsa_prefix_cache* dsa_prefix_cache_create(int32_t page_size, int32_t num_pages) {
  if (page_size <= 0 || num_pages <= 0) return nullptr;
  dsa_prefix_cache* c = new (std::nothrow) dsa_prefix_cache();
  if (!c) return nullptr;
  try {
    c->page_size = page_size;
    c->num_pages = num_pages;
    c->node_of.assign(num_pages, nullptr);
    c->priv_refs.assign(num_pages, 0);
    c->free_list.reserve(num_pages);
    for (int32_t p = num_pages - 1; p >= 0; --p) c->free_list.push_back(p);  // hands out 0, 1, 2, ...
  } catch (...) {
    delete c;
    return nullptr;
  }
  return c;
}

void dsa_prefix_cache_destroy(dsa_prefix_cache* c) {
  if (!c) return;
  std::vector<Node*> stack;
  for (auto& kv : c->root.kids) stack.push_back(kv.second);
  while (!stack.empty()) {
    Node* n = stack.back();
    stack.pop_back();
    for (auto& kv : n->kids) stack.push_back(kv.second);
    delete n;
  }
  delete c;
}

dsa_status dsa_prefix_cache_acquire(dsa_prefix_cache* c, const int32_t* tokens, int64_t n_tokens,
                                    int32_t* block_table, int32_t max_pages, int32_t* n_pages, int32_t* n_shared) {
  if (!c || n_tokens < 0 || (n_tokens > 0 && (!tokens || !block_table)) || max_pages < 0) return DSA_ERR_INVALID_ARG;
  const int32_t P = c->page_size;
  const int64_t need = (n_tokens + P - 1) / P;
  if (need > max_pages) return DSA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(c->mu);
  const int64_t full = n_tokens / P;
  // 1. the longest cached prefix of whole pages
  Node* at = &c->root;
  int64_t shared = 0;
  std::vector<Node*> path;
  while (shared < full) {
    Node* k = c->find_child(at, tokens + shared * P);
    if (!k) break;
    path.push_back(k);
    at = k;
    ++shared;
  }
  // 2. fresh pages for the rest: reference the shared ones first so that
  //    eviction cannot take them, and give everything back on failure
  for (Node* n : path) c->ref_node(n);
  std::vector<int32_t> fresh;
  for (int64_t p = shared; p < need; ++p) {
    const int32_t pg = c->take_page();
    if (pg < 0) {
      for (int32_t f : fresh) c->free_list.push_back(f);
      for (Node* n : path) c->unref_node(n);
      return DSA_ERR_OUT_OF_PAGES;
    }
    fresh.push_back(pg);
  }
  // 3. the request's new full pages join the tree; a partial last page stays private
  for (int64_t p = 0; p < shared; ++p) block_table[p] = path[p]->page;
  for (int64_t p = shared; p < need; ++p) {
    const int32_t pg = fresh[p - shared];
    block_table[p] = pg;
    if (p < full) {
      Node* n = new Node();
      n->page = pg;
      n->parent = at;
      n->tokens.assign(tokens + p * P, tokens + (p + 1) * P);
      c->unmark(at);  // no longer a leaf
      at->kids.emplace(hash_tokens(n->tokens.data(), P), n);
      c->node_of[pg] = n;
      ++c->cached;
      c->ref_node(n);
      at = n;
    } else {
      c->priv_refs[pg] = 1;
      ++c->referenced;
    }
  }
  if (n_pages) *n_pages = (int32_t)need;
  if (n_shared) *n_shared = (int32_t)shared;
  return DSA_OK;
}

dsa_status dsa_prefix_cache_release(dsa_prefix_cache* c, const int32_t* block_table, int32_t n_pages) {
  if (!c || n_pages < 0 || (n_pages > 0 && !block_table)) return DSA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(c->mu);
  for (int32_t i = 0; i < n_pages; ++i) {
    const int32_t pg = block_table[i];
    if (pg < 0 || pg >= c->num_pages) return DSA_ERR_INVALID_ARG;
    if (!c->node_of[pg] && c->priv_refs[pg] <= 0) return DSA_ERR_INVALID_ARG;
    if (c->node_of[pg] && c->node_of[pg]->refs <= 0) return DSA_ERR_INVALID_ARG;
  }
  // the deepest pages first, so that a released leaf is marked before its parent
  for (int32_t i = n_pages - 1; i >= 0; --i) {
    const int32_t pg = block_table[i];
    if (Node* n = c->node_of[pg]) {
      c->unref_node(n);
    } else if (--c->priv_refs[pg] == 0) {
      --c->referenced;
      c->free_list.push_back(pg);
    }
  }
  return DSA_OK;
}

dsa_status dsa_prefix_cache_stats(dsa_prefix_cache* c, int32_t* pages_referenced, int32_t* pages_cached,
                                  int32_t* pages_free) {
  if (!c) return DSA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(c->mu);
  if (pages_referenced) *pages_referenced = c->referenced;
  if (pages_cached) *pages_cached = c->cached;
  if (pages_free) *pages_free = (int32_t)c->free_list.size();
  return DSA_OK;
}

}  // extern "C"
