// Host-side KV page pool and radix prefix tree.
//
// Prefix sharing follows "SGLang Day-0 Support for FishAudio S2"
// (Optimizations with SGLang Omni: radix prefix caching keeps the KV of a
// shared system prompt / reference audio across requests) and "Fish Audio
// Abre Codigo do S2" (Streaming de Produção via SGLang: reference-audio
// tokens in the system prompt hit the prefix cache).  Sharing is in whole
// 16-position pages; a position's key is (token, mask, and the codebook codes
// when masked), since the codes are part of what the position feeds the
// model.
#pragma once

#include <stdint.h>

#include <algorithm>
#include <cstring>
#include <unordered_map>
#include <vector>

namespace s2 {

constexpr int kKeyInts = 12;  // token, mask, 10 codes

class PagePool {
 public:
  void init(int n_pages, uint64_t perm_seed) {
    ref_.assign(n_pages, 0);
    free_.clear();
    std::vector<int> order(n_pages);
    for (int i = 0; i < n_pages; ++i) order[i] = i;
    if (perm_seed) {  // Fisher-Yates with splitmix64
      uint64_t s = perm_seed;
      for (int i = n_pages - 1; i > 0; --i) {
        s += 0x9E3779B97F4A7C15ull;
        uint64_t z = s;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        z ^= z >> 31;
        int j = (int)(z % (uint64_t)(i + 1));
        int t = order[i]; order[i] = order[j]; order[j] = t;
      }
    }
    for (int i = n_pages - 1; i >= 0; --i) free_.push_back(order[i]);  // pop_back gives order[0] first
  }
  int n_free() const { return (int)free_.size(); }
  int n_total() const { return (int)ref_.size(); }
  int ref(int p) const { return ref_[p]; }
  int alloc() {
    int p = free_.back();
    free_.pop_back();
    ref_[p] = 1;
    return p;
  }
  void incref(int p) { ++ref_[p]; }
  void decref(int p) {
    if (--ref_[p] == 0) free_.push_back(p);
  }

 private:
  std::vector<int> ref_;
  std::vector<int> free_;
};

class RadixTree {
 public:
  explicit RadixTree(int page = 16) : page_(page) { nodes_.push_back(Node{}); }

  // Pages of the longest cached page-aligned prefix of ``keys`` (n_pos
  // positions of kKeyInts ints), at most max_pages.
  std::vector<int> match(const std::vector<int32_t>& keys, int n_pos, int max_pages) {
    std::vector<int> out;
    int node = 0;
    const int n_full = n_pos / page_;
    ++tick_;
    for (int i = 0; i < n_full && i < max_pages; ++i) {
      int nxt = child(node, keys.data() + (size_t)i * page_ * kKeyInts);
      if (nxt < 0) break;
      out.push_back(nodes_[nxt].page);
      nodes_[nxt].last_use = tick_;
      node = nxt;
    }
    return out;
  }

  // Least-recently-used eviction: drop leaf pages that only the tree still
  // references (pool ref count 1), oldest first, until ``want`` pages are
  // gathered or none is left.  Returns the dropped pages (the caller
  // releases the tree's reference on each).
  std::vector<int> evict(int want, const PagePool& pool) {
    std::vector<int> out;
    while ((int)out.size() < want) {
      std::vector<std::pair<uint64_t, int>> leaves;
      for (int i = 1; i < (int)nodes_.size(); ++i) {
        const Node& n = nodes_[i];
        if (!n.dead && n.kids.empty() && pool.ref(n.page) == 1) leaves.push_back({n.last_use, i});
      }
      if (leaves.empty()) break;
      std::sort(leaves.begin(), leaves.end());
      for (auto& lv : leaves) {
        if ((int)out.size() >= want) break;
        Node& n = nodes_[lv.second];
        auto& sib = nodes_[n.parent].kids[n.h];
        sib.erase(std::remove(sib.begin(), sib.end(), lv.second), sib.end());
        if (sib.empty()) nodes_[n.parent].kids.erase(n.h);
        n.dead = true;
        out.push_back(n.page);
        --held_;
        ++dead_;
      }
    }
    if (dead_ > 64 && 2 * dead_ > (int)nodes_.size()) compact();
    return out;
  }

  // Pages evict() could drop in all: nodes whose page, and every page below
  // them, only the tree references (a child is always stored after its
  // parent, so one backward pass sees the children first).
  int evictable(const PagePool& pool) const {
    std::vector<char> blocked(nodes_.size(), 0);
    int n = 0;
    for (int i = (int)nodes_.size() - 1; i >= 1; --i) {
      const Node& nd = nodes_[i];
      if (nd.dead) continue;
      if (!blocked[i] && pool.ref(nd.page) == 1) ++n;
      else blocked[nd.parent] = 1;
    }
    return n;
  }

  // Record the full pages of ``keys``; returns the pages newly held.
  std::vector<int> insert(const std::vector<int32_t>& keys, int n_pos, const std::vector<int>& pages) {
    std::vector<int> added;
    ++tick_;
    int node = 0;
    const int n_full = std::min<int>(n_pos / page_, (int)pages.size());
    for (int i = 0; i < n_full; ++i) {
      const int32_t* k = keys.data() + (size_t)i * page_ * kKeyInts;
      int nxt = child(node, k);
      if (nxt < 0) {
        Node n;
        n.page = pages[i];
        n.key.assign(k, k + (size_t)page_ * kKeyInts);
        n.parent = node;
        n.h = hash(k);
        nxt = (int)nodes_.size();
        nodes_.push_back(std::move(n));
        nodes_[node].kids[nodes_[nxt].h].push_back(nxt);
        added.push_back(pages[i]);
      }
      nodes_[nxt].last_use = tick_;
      node = nxt;
    }
    held_ += (int)added.size();
    return added;
  }
  int held() const { return held_; }
  int page() const { return page_; }

  // Pages the tree holds a reference on, in node order.
  std::vector<int> pages() const {
    std::vector<int> out;
    for (size_t i = 1; i < nodes_.size(); ++i)
      if (!nodes_[i].dead) out.push_back(nodes_[i].page);
    return out;
  }

  // Drop every node; returns the pages the tree held.
  std::vector<int> clear() {
    std::vector<int> pages;
    for (size_t i = 1; i < nodes_.size(); ++i)
      if (!nodes_[i].dead) pages.push_back(nodes_[i].page);
    nodes_.clear();
    nodes_.push_back(Node{});
    held_ = 0;
    dead_ = 0;
    return pages;
  }

  // Nodes stored, live or dropped (the root included).
  int stored() const { return (int)nodes_.size(); }

 private:
  struct Node {
    int page = -1;
    int parent = -1;
    uint64_t h = 0;
    uint64_t last_use = 0;
    bool dead = false;
    std::vector<int32_t> key;
    std::unordered_map<uint64_t, std::vector<int>> kids;
  };
  uint64_t hash(const int32_t* k) const {
    uint64_t h = 1469598103934665603ull;
    for (int i = 0; i < page_ * kKeyInts; ++i) {
      h ^= (uint32_t)k[i];
      h *= 1099511628211ull;
    }
    return h;
  }
  int child(int node, const int32_t* k) const {
    auto it = nodes_[node].kids.find(hash(k));
    if (it == nodes_[node].kids.end()) return -1;
    for (int c : it->second)
      if (std::memcmp(nodes_[c].key.data(), k, sizeof(int32_t) * page_ * kKeyInts) == 0) return c;
    return -1;
  }
  // Remove dropped nodes, keeping the stored order: a parent still precedes
  // its children and older nodes precede newer ones (the eviction tie-break).
  // A dropped node was a leaf, so no live node refers to one.
  void compact() {
    std::vector<int> remap(nodes_.size(), -1);
    int k = 0;
    for (size_t i = 0; i < nodes_.size(); ++i)
      if (i == 0 || !nodes_[i].dead) remap[i] = k++;
    std::vector<Node> kept;
    kept.reserve(k);
    for (size_t i = 0; i < nodes_.size(); ++i) {
      if (remap[i] < 0) continue;
      Node n = std::move(nodes_[i]);
      if (n.parent >= 0) n.parent = remap[n.parent];
      for (auto& kv : n.kids)
        for (int& c : kv.second) c = remap[c];
      kept.push_back(std::move(n));
    }
    nodes_.swap(kept);
    dead_ = 0;
  }

  int page_;
  int held_ = 0;
  int dead_ = 0;
  uint64_t tick_ = 0;
  std::vector<Node> nodes_;
};

// Cache keys of a prompt's T positions: token, mask flag, and the NC codebook
// codes (codes laid out [NC][T]) when the position is masked, else zeros.
inline void position_keys(const int32_t* tok, const int32_t* codes, const uint8_t* mask, int T, int NC,
                          std::vector<int32_t>& keys) {
  keys.assign((size_t)T * kKeyInts, 0);
  for (int t = 0; t < T; ++t) {
    int32_t* k = keys.data() + (size_t)t * kKeyInts;
    k[0] = tok[t];
    const int m = mask ? (mask[t] != 0) : 0;
    k[1] = m;
    if (m)
      for (int j = 0; j < NC; ++j) k[2 + j] = codes[(size_t)j * T + t];
  }
}

// Free pages until ``need`` are available, dropping least-recently-used leaves
// that only the tree still references (no tree: nothing to drop).  When even
// every droppable page would not be enough, nothing is dropped, so a call that
// then fails for lack of pages leaves the cache as it was.  Returns the number
// of pages dropped; the caller checks n_free() afterwards.
inline int make_room(PagePool& pool, RadixTree* tree, int need) {
  int dropped = 0;
  if (tree && need > pool.n_free() && need - pool.n_free() <= tree->evictable(pool))
    for (int pg : tree->evict(need - pool.n_free(), pool)) {
      pool.decref(pg);
      ++dropped;
    }
  return dropped;
}

// Grow page tables so that table i covers want[i] positions (page-sized
// positions per page): the pages missing over all tables are counted first,
// room is made as make_room does, and only if the pool can then supply all of
// them is any allocated (in table order).  Returns false, with nothing
// allocated, when it cannot; *dropped gets the pages dropped from the tree.
inline bool reserve_pages(PagePool& pool, RadixTree* tree, const std::vector<std::vector<int>*>& tables,
                          const std::vector<int>& want, int page, int* dropped) {
  int need = 0;
  for (size_t i = 0; i < tables.size(); ++i)
    need += std::max(0, (want[i] + page - 1) / page - (int)tables[i]->size());
  const int d = make_room(pool, tree, need);
  if (dropped) *dropped = d;
  if (need > pool.n_free()) return false;
  for (size_t i = 0; i < tables.size(); ++i)
    while ((int)tables[i]->size() * page < want[i]) tables[i]->push_back(pool.alloc());
  return true;
}

// Page table for a new prompt of T positions (keys from position_keys): the
// longest cached page-aligned prefix that leaves at least one position to
// compute (its pages pinned with one more reference each), then fresh pages
// for the rest.  Returns the number of cached positions, or -1 with nothing
// held when the pool cannot supply the fresh pages even after eviction.
inline int admit_prompt(PagePool& pool, RadixTree* tree, const std::vector<int32_t>& keys, int T,
                        std::vector<int>& table, int* dropped) {
  const int P = tree ? tree->page() : 16;
  std::vector<int> hit;
  if (tree) hit = tree->match(keys, T, (T - 1) / P);
  const int need = (T + P - 1) / P - (int)hit.size();
  for (int pg : hit) pool.incref(pg);  // pinned before any eviction
  const int d = make_room(pool, tree, need);
  if (dropped) *dropped = d;
  if (need > pool.n_free()) {
    for (int pg : hit) pool.decref(pg);
    return -1;
  }
  table = hit;
  for (int i = 0; i < need; ++i) table.push_back(pool.alloc());
  return (int)hit.size() * P;
}

}  // namespace s2
