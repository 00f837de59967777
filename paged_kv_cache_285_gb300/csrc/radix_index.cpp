// Host prefix index of the paged cache: a radix tree over token ids whose
// edges own whole KV blocks, with leaf-first LRU eviction.
//
// "PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화", section 03: the
// KV states of finished requests are kept on token paths of a radix tree
// (common prefixes stored once); a new request takes the longest matching
// path, reuses its KV and prefills only the rest (figure: inserting "firm"
// next to dog, dot, pump, fat, fire reuses f-i-r and adds m).  When memory
// runs short, leaf branches are evicted first, least recently used first,
// so interior prefixes shared by many requests survive (section 03, LRU
// figure).  With paged KV only whole blocks can be shared, so every edge
// label is a whole number of blocks and a match is a whole number of blocks.
//
// The index also owns the pool of physical block ids [0, num_blocks): a block
// is free, held by a caller (allocated, not yet inserted), or held by the tree.
// Not thread-safe: one caller at a time.
#include <algorithm>
#include <cstdint>
#include <map>
#include <memory>
#include <new>
#include <set>
#include <utility>
#include <vector>

#include "../../include/pkv.h"

namespace {

enum : uint8_t { kFree = 0, kCaller = 1, kTree = 2 };

// One block of token ids, viewed in place (a lookup key that allocates nothing).
struct BlockView {
  const int32_t* p;
  int32_t n;
};

// Lexicographic order of token blocks, comparable across stored keys and views.
struct BlockLess {
  using is_transparent = void;
  static bool less(const int32_t* a, size_t na, const int32_t* b, size_t nb) {
    return std::lexicographical_compare(a, a + na, b, b + nb);
  }
  bool operator()(const std::vector<int32_t>& a, const std::vector<int32_t>& b) const {
    return less(a.data(), a.size(), b.data(), b.size());
  }
  bool operator()(const std::vector<int32_t>& a, const BlockView& b) const {
    return less(a.data(), a.size(), b.p, (size_t)b.n);
  }
  bool operator()(const BlockView& a, const std::vector<int32_t>& b) const {
    return less(a.p, (size_t)a.n, b.data(), b.size());
  }
};

struct Node {
  std::vector<int32_t> tokens;  // edge label: a whole number of blocks of token ids
  std::vector<int32_t> blocks;  // physical block of each block of the label
  std::map<std::vector<int32_t>, std::unique_ptr<Node>, BlockLess> children;  // by first block
  Node* parent = nullptr;
  uint64_t last_use = 0;
  int64_t locks = 0;
  bool listed = false;  // in the evictable set under key (listed_use, this)
  uint64_t listed_use = 0;
};

}  // namespace

struct pkv_radix_index {
  int32_t bs = 0;
  int32_t num_blocks = 0;
  Node root;
  std::vector<int32_t> free_list;
  std::vector<uint8_t> state;
  uint64_t clock = 0;
  int64_t nodes = 0;
  int64_t tree_blocks = 0;
  std::set<std::pair<uint64_t, Node*>> evictable;  // unlocked leaves, least recently used first

  BlockView key_at(const int32_t* tokens, int64_t blk) const { return {tokens + blk * bs, bs}; }

  // Keep a node's entry in the evictable set in step with its state.
  void refresh(Node* n) {
    if (n == &root) return;
    if (n->listed) {
      evictable.erase({n->listed_use, n});
      n->listed = false;
    }
    if (n->children.empty() && n->locks == 0) {
      n->listed_use = n->last_use;
      evictable.insert({n->listed_use, n});
      n->listed = true;
    }
  }

  // Split n's edge after its first k blocks (0 < k < blocks); returns the new
  // upper node, which takes n's place under its parent.
  Node* split(Node* n, int64_t k) {
    auto mid = std::make_unique<Node>();
    Node* m = mid.get();
    m->tokens.assign(n->tokens.begin(), n->tokens.begin() + k * bs);
    m->blocks.assign(n->blocks.begin(), n->blocks.begin() + k);
    m->parent = n->parent;
    m->last_use = n->last_use;
    m->locks = n->locks;  // every lock through n also runs through m
    Node* parent = n->parent;
    auto& slot = parent->children.find(key_at(n->tokens.data(), 0))->second;
    std::unique_ptr<Node> lower = std::move(slot);
    lower->tokens.erase(lower->tokens.begin(), lower->tokens.begin() + k * bs);
    lower->blocks.erase(lower->blocks.begin(), lower->blocks.begin() + k);
    lower->parent = m;
    std::vector<int32_t> lower_key(lower->tokens.begin(), lower->tokens.begin() + bs);
    m->children.emplace(std::move(lower_key), std::move(lower));
    slot = std::move(mid);
    ++nodes;
    refresh(m);
    return m;
  }

  // Follow tokens [0, nblk blocks) from the root, splitting the edge where the
  // path diverges inside it; returns the deepest node reached and the number
  // of blocks it covers.  The path from the root to that node is returned in
  // `path` when non-null.
  std::pair<Node*, int64_t> walk(const int32_t* tokens, int64_t nblk, std::vector<Node*>* path) {
    Node* cur = &root;
    int64_t i = 0;
    while (i < nblk) {
      auto it = cur->children.find(key_at(tokens, i));
      if (it == cur->children.end()) break;
      Node* child = it->second.get();
      const int64_t nb = (int64_t)child->blocks.size();
      int64_t m = 1;
      while (m < nb && i + m < nblk &&
             std::equal(child->tokens.begin() + m * bs, child->tokens.begin() + (m + 1) * bs,
                        tokens + (i + m) * bs))
        ++m;
      if (m < nb) child = split(child, m);
      if (path) path->push_back(child);
      cur = child;
      i += m;
    }
    return {cur, i};
  }

  void touch(Node* n) {
    n->last_use = ++clock;
    refresh(n);
  }

  bool evict_one() {
    if (evictable.empty()) return false;
    Node* n = evictable.begin()->second;
    evictable.erase(evictable.begin());
    n->listed = false;
    for (int32_t b : n->blocks) {
      state[b] = kFree;
      free_list.push_back(b);
    }
    tree_blocks -= (int64_t)n->blocks.size();
    Node* parent = n->parent;
    parent->children.erase(parent->children.find(key_at(n->tokens.data(), 0)));
    --nodes;
    refresh(parent);
    return true;
  }
};

extern "C" {

pkv_status pkv_radix_create(int32_t block_size, int32_t num_blocks, pkv_radix_index** out) {
  if (!out || block_size <= 0 || num_blocks < 0) return PKV_ERR_INVALID_ARG;
  *out = nullptr;
  pkv_radix_index* x = new (std::nothrow) pkv_radix_index();
  if (!x) return PKV_ERR_NO_SPACE;
  x->bs = block_size;
  x->num_blocks = num_blocks;
  x->state.assign((size_t)num_blocks, kFree);
  x->free_list.reserve((size_t)num_blocks);
  for (int32_t b = num_blocks - 1; b >= 0; --b) x->free_list.push_back(b);  // hand out 0, 1, ...
  *out = x;
  return PKV_OK;
}

void pkv_radix_destroy(pkv_radix_index* x) { delete x; }

pkv_status pkv_radix_match(pkv_radix_index* x, const int32_t* tokens, int32_t num_tokens,
                           int32_t* blocks_out, int32_t blocks_cap, int32_t* matched_tokens) {
  if (!x || num_tokens < 0 || (num_tokens > 0 && !tokens) || !matched_tokens || blocks_cap < 0)
    return PKV_ERR_INVALID_ARG;
  const int64_t nblk = num_tokens / x->bs;
  std::vector<Node*> path;
  const auto r = x->walk(tokens, nblk, &path);
  if (r.second > blocks_cap || (r.second > 0 && !blocks_out)) {
    // the caller's buffer cannot hold the matched blocks: nothing is locked
    *matched_tokens = (int32_t)(r.second * x->bs);
    return PKV_ERR_INVALID_ARG;
  }
  int64_t k = 0;
  for (Node* n : path) {
    for (int32_t b : n->blocks) blocks_out[k++] = b;
    ++n->locks;
    x->touch(n);
  }
  *matched_tokens = (int32_t)(r.second * x->bs);
  return PKV_OK;
}

pkv_status pkv_radix_release(pkv_radix_index* x, const int32_t* tokens, int32_t matched_tokens) {
  if (!x || matched_tokens < 0 || matched_tokens % x->bs != 0 || (matched_tokens > 0 && !tokens))
    return PKV_ERR_INVALID_ARG;
  const int64_t nblk = matched_tokens / x->bs;
  // the matched path still ends on a node boundary (splits only add
  // boundaries, and locked nodes are never evicted)
  std::vector<Node*> path;
  Node* cur = &x->root;
  int64_t i = 0;
  while (i < nblk) {
    auto it = cur->children.find(x->key_at(tokens, i));
    if (it == cur->children.end()) return PKV_ERR_INVALID_ARG;
    Node* child = it->second.get();
    const int64_t nb = (int64_t)child->blocks.size();
    if (i + nb > nblk || child->locks <= 0 ||
        !std::equal(child->tokens.begin(), child->tokens.end(), tokens + i * x->bs))
      return PKV_ERR_INVALID_ARG;
    path.push_back(child);
    cur = child;
    i += nb;
  }
  for (Node* n : path) {
    --n->locks;
    x->touch(n);
  }
  return PKV_OK;
}

pkv_status pkv_radix_alloc(pkv_radix_index* x, int32_t count, int32_t* blocks_out) {
  if (!x || count < 0 || (count > 0 && !blocks_out)) return PKV_ERR_INVALID_ARG;
  while ((int64_t)x->free_list.size() < count)
    if (!x->evict_one()) return PKV_ERR_NO_SPACE;
  for (int32_t k = 0; k < count; ++k) {
    const int32_t b = x->free_list.back();
    x->free_list.pop_back();
    x->state[b] = kCaller;
    blocks_out[k] = b;
  }
  return PKV_OK;
}

pkv_status pkv_radix_free(pkv_radix_index* x, const int32_t* blocks, int32_t count) {
  if (!x || count < 0 || (count > 0 && !blocks)) return PKV_ERR_INVALID_ARG;
  for (int32_t k = 0; k < count; ++k) {
    const int32_t b = blocks[k];
    if (b < 0 || b >= x->num_blocks || x->state[b] != kCaller) return PKV_ERR_INVALID_ARG;
  }
  for (int32_t k = 0; k < count; ++k) {
    x->state[blocks[k]] = kFree;
    x->free_list.push_back(blocks[k]);
  }
  return PKV_OK;
}

pkv_status pkv_radix_insert(pkv_radix_index* x, const int32_t* tokens, int32_t num_tokens,
                            const int32_t* blocks, int32_t* released_out, int32_t* num_released) {
  if (!x || num_tokens < 0 || (num_tokens > 0 && (!tokens || !blocks)) || !num_released)
    return PKV_ERR_INVALID_ARG;
  const int64_t nblk = num_tokens / x->bs;
  // every full block the caller passes is either the tree's own (it matched
  // it) or held by the caller
  std::vector<Node*> path;
  for (int64_t k = 0; k < nblk; ++k) {
    const int32_t b = blocks[k];
    if (b < 0 || b >= x->num_blocks || x->state[b] == kFree) return PKV_ERR_INVALID_ARG;
  }
  const auto r = x->walk(tokens, nblk, &path);
  // Check everything before changing any state: blocks of the part the tree
  // already holds are either the tree's own (the caller matched them) or the
  // caller's, which go back to the pool; the rest must be the caller's, and no
  // caller block may appear twice.
  std::vector<int32_t> tree_of(nblk, -1);
  {
    int64_t k = 0;
    for (Node* n : path)
      for (int32_t tb : n->blocks) tree_of[k++] = tb;
  }
  std::vector<int32_t> mine;
  for (int64_t q = 0; q < nblk; ++q) {
    const int32_t cb = blocks[q];
    if (q < r.second && cb == tree_of[q]) continue;
    if (x->state[cb] != kCaller) return PKV_ERR_INVALID_ARG;
    mine.push_back(cb);
  }
  std::sort(mine.begin(), mine.end());
  if (std::adjacent_find(mine.begin(), mine.end()) != mine.end()) return PKV_ERR_INVALID_ARG;
  int32_t nrel = 0;
  for (int64_t q = 0; q < r.second; ++q) {
    const int32_t cb = blocks[q];
    if (cb == tree_of[q]) continue;
    x->state[cb] = kFree;
    x->free_list.push_back(cb);
    if (released_out) released_out[nrel] = cb;
    ++nrel;
  }
  for (Node* n : path) x->touch(n);
  if (r.second < nblk) {
    auto leaf = std::make_unique<Node>();
    Node* l = leaf.get();
    l->tokens.assign(tokens + r.second * x->bs, tokens + nblk * x->bs);
    l->blocks.assign(blocks + r.second, blocks + nblk);
    for (int32_t b : l->blocks) x->state[b] = kTree;
    x->tree_blocks += nblk - r.second;
    l->parent = r.first;
    r.first->children.emplace(
        std::vector<int32_t>(tokens + r.second * x->bs, tokens + (r.second + 1) * x->bs),
        std::move(leaf));
    ++x->nodes;
    x->refresh(r.first);
    x->touch(l);
  }
  *num_released = nrel;
  return PKV_OK;
}

pkv_status pkv_radix_evict(pkv_radix_index* x, int32_t num_blocks, int32_t* freed) {
  if (!x || num_blocks < 0 || !freed) return PKV_ERR_INVALID_ARG;
  const int64_t before = (int64_t)x->free_list.size();
  while ((int64_t)x->free_list.size() - before < num_blocks && x->evict_one()) {
  }
  *freed = (int32_t)((int64_t)x->free_list.size() - before);
  return PKV_OK;
}

pkv_status pkv_radix_stats(const pkv_radix_index* x, pkv_radix_stats_t* out) {
  if (!x || !out) return PKV_ERR_INVALID_ARG;
  out->num_blocks = x->num_blocks;
  out->free_blocks = (int32_t)x->free_list.size();
  out->tree_blocks = (int32_t)x->tree_blocks;
  out->caller_blocks = x->num_blocks - out->free_blocks - out->tree_blocks;
  out->nodes = (int32_t)x->nodes;
  out->evictable_leaves = (int32_t)x->evictable.size();
  return PKV_OK;
}

}  // extern "C"
