// Host block pool with prefix caching: the allocator that produces the block
// tables and slot mappings the kernels consume.  Declarations, ownership and
// error conventions are in include/pagedkv.h.
//
// Sources ("第34讲 … vLLM 生产级系统架构全景剖析与四重加速引擎"):
//  §1.2  KVCacheManager.allocate_slots fills a request's last block before
//        taking a new one; free(req) releases blocks tail first.  BlockPool
//        keeps free blocks in a doubly linked queue (FreeKVCacheBlockQueue) so
//        that a cached block can leave it from the middle in O(1).
//  §2.2  a new request reuses the longest cached prefix, in whole blocks, and
//        each reused block gains a reference.
//  §2.3  blocks reaching ref_cnt 0 keep their data and join the queue's tail;
//        allocation takes the head, evicting whatever prefix it held.
//  openeuler.csdn.net PagedAttention notes, "机制 2：写时复制": a forked request
//  shares blocks by reference; writing into a shared block first copies it.
//
// Layout: the queue is intrusive (prev/next arrays, sentinel num_blocks).  A
// cached block is found by a 128-bit chained hash of its token prefix (the
// parent block's hash and the block's own tokens) and confirmed by comparing
// its stored tokens, so a false hit needs two different earlier prefixes with
// equal 128-bit hashes.  Not thread-safe: callers serialise access to a pool.

#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"

namespace {

struct Key {
  uint64_t a, b;
  bool operator==(const Key& o) const { return a == o.a && b == o.b; }
};
struct KeyHash {
  size_t operator()(const Key& k) const { return (size_t)(k.a ^ (k.b >> 7)); }
};

// Finaliser of the SplitMix64 generator (Steele, Lea and Flood, "Fast
// splittable pseudorandom number generators", OOPSLA 2014).
inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

// The empty prefix, then one step per full block.
constexpr Key kRoot = {0x243f6a8885a308d3ull, 0x13198a2e03707344ull};

Key chain(const Key& parent, const int32_t* toks, int n) {
  uint64_t a = parent.a, b = parent.b;
  for (int i = 0; i < n; ++i) {
    const uint64_t t = (uint32_t)toks[i];
    a = mix64(a ^ (t + 0x9e3779b97f4a7c15ull));
    b = mix64(b + t * 0xc2b2ae3d27d4eb4full + 0x165667b19e3779f9ull);
  }
  return {a, b};
}

}  // namespace

struct pkv_block_pool {
  int32_t nb = 0, bs = 0, nfree = 0;
  std::vector<int32_t> prev, next;  // free queue; index nb is the sentinel
  std::vector<int32_t> ref;
  std::vector<uint8_t> cached;
  std::vector<Key> key;        // of cached blocks
  std::vector<int32_t> toks;   // nb x bs tokens of cached blocks
  std::unordered_map<Key, int32_t, KeyHash> map;

  void push_back(int32_t id) {
    const int32_t last = prev[nb];
    next[last] = id;
    prev[id] = last;
    next[id] = nb;
    prev[nb] = id;
    ++nfree;
  }
  void unlink(int32_t id) {
    next[prev[id]] = next[id];
    prev[next[id]] = prev[id];
    prev[id] = next[id] = -1;
    --nfree;
  }
  // a reference to a block that may sit in the queue
  void take(int32_t id) {
    if (ref[id]++ == 0) unlink(id);
  }
  // the queue's head, its cached prefix evicted
  int32_t alloc() {
    const int32_t id = next[nb];
    unlink(id);
    if (cached[id]) {
      map.erase(key[id]);
      cached[id] = 0;
    }
    ref[id] = 1;
    return id;
  }
  void release(int32_t id) {
    if (--ref[id] == 0) push_back(id);
  }
  bool same_tokens(int32_t id, const int32_t* t) const {
    return std::memcmp(&toks[(size_t)id * bs], t, sizeof(int32_t) * bs) == 0;
  }
};

struct pkv_request {
  pkv_block_pool* pool = nullptr;
  std::vector<int32_t> table;
  int32_t ntok = 0;
  Key last = kRoot;              // chain through the last full block
  std::vector<int32_t> partial;  // tokens of the partial last block
};

extern "C" {

int pkv_block_pool_create(int32_t num_blocks, int32_t block_size, pkv_block_pool** out) {
  if (!out) return PKV_ERR_INVALID_ARG;
  *out = nullptr;
  if (num_blocks < 0 || block_size <= 0 || (int64_t)num_blocks * block_size > (1ll << 40))
    return PKV_ERR_INVALID_ARG;
  pkv_block_pool* p = new (std::nothrow) pkv_block_pool;
  if (!p) return PKV_ERR_INVALID_ARG;
  try {
    p->nb = num_blocks;
    p->bs = block_size;
    p->prev.assign(num_blocks + 1, -1);
    p->next.assign(num_blocks + 1, -1);
    p->prev[num_blocks] = p->next[num_blocks] = num_blocks;
    p->ref.assign(num_blocks, 0);
    p->cached.assign(num_blocks, 0);
    p->key.assign(num_blocks, Key{0, 0});
    p->toks.assign((size_t)num_blocks * block_size, 0);
    for (int32_t i = 0; i < num_blocks; ++i) p->push_back(i);
  } catch (...) {
    delete p;
    return PKV_ERR_INVALID_ARG;
  }
  *out = p;
  return PKV_OK;
}

void pkv_block_pool_destroy(pkv_block_pool* pool) { delete pool; }

int32_t pkv_block_pool_num_free(const pkv_block_pool* pool) { return pool ? pool->nfree : -1; }

int32_t pkv_block_pool_num_cached(const pkv_block_pool* pool) {
  return pool ? (int32_t)pool->map.size() : -1;
}

int32_t pkv_block_pool_ref_cnt(const pkv_block_pool* pool, int32_t block) {
  if (!pool || block < 0 || block >= pool->nb) return -1;
  return pool->ref[block];
}

int32_t pkv_block_pool_is_cached(const pkv_block_pool* pool, int32_t block) {
  if (!pool || block < 0 || block >= pool->nb) return -1;
  return pool->cached[block];
}

int32_t pkv_block_pool_queue(const pkv_block_pool* pool, int32_t* out, int32_t max) {
  if (!pool) return -1;
  int32_t n = 0;
  for (int32_t id = pool->next[pool->nb]; id != pool->nb; id = pool->next[id], ++n)
    if (out && n < max) out[n] = id;
  return n;
}

int pkv_request_create(pkv_block_pool* pool, pkv_request** out) {
  if (!out) return PKV_ERR_INVALID_ARG;
  *out = nullptr;
  if (!pool) return PKV_ERR_INVALID_ARG;
  pkv_request* r = new (std::nothrow) pkv_request;
  if (!r) return PKV_ERR_INVALID_ARG;
  r->pool = pool;
  *out = r;
  return PKV_OK;
}

int pkv_request_match_prefix(pkv_request* req, const int32_t* tokens, int32_t num_tokens,
                             int32_t* matched_out) {
  if (!req || (num_tokens > 0 && !tokens) || num_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (req->ntok != 0 || !req->table.empty()) return PKV_ERR_INVALID_ARG;
  pkv_block_pool* p = req->pool;
  const int32_t bs = p->bs;
  Key h = kRoot;
  int32_t matched = 0;
  for (int32_t end = bs; end <= num_tokens - 1; end += bs) {
    const Key k = chain(h, tokens + end - bs, bs);
    const auto it = p->map.find(k);
    if (it == p->map.end() || !p->same_tokens(it->second, tokens + end - bs)) break;
    p->take(it->second);
    req->table.push_back(it->second);
    h = k;
    matched = end;
  }
  req->ntok = matched;
  req->last = h;
  if (matched_out) *matched_out = matched;
  return PKV_OK;
}

int pkv_request_append(pkv_request* req, const int32_t* token_ids, int32_t num_tokens,
                       int64_t* slots_out, int32_t* cow_out) {
  if (!req || num_tokens < 0 || (num_tokens > 0 && !token_ids)) return PKV_ERR_INVALID_ARG;
  if (cow_out) cow_out[0] = cow_out[1] = -1;
  if (num_tokens == 0) return PKV_OK;
  pkv_block_pool* p = req->pool;
  const int32_t bs = p->bs, t0 = req->ntok;
  if ((int64_t)t0 + num_tokens > (int64_t)1 << 30) return PKV_ERR_INVALID_ARG;
  const bool cow = t0 % bs != 0 && p->ref[req->table.back()] > 1;
  const int64_t need = (cow ? 1 : 0) + ((int64_t)t0 + num_tokens + bs - 1) / bs -
                       ((int64_t)t0 + bs - 1) / bs;
  if (need > p->nfree) return PKV_ERR_NO_BLOCKS;
  if (cow) {
    const int32_t old = req->table.back();
    const int32_t id = p->alloc();
    p->release(old);
    req->table.back() = id;
    if (cow_out) {
      cow_out[0] = old;
      cow_out[1] = id;
    }
  }
  for (int32_t i = 0; i < num_tokens; ++i) {
    const int32_t pos = t0 + i;
    if (pos % bs == 0) req->table.push_back(p->alloc());
    const int32_t id = req->table[pos / bs];
    if (slots_out) slots_out[i] = (int64_t)id * bs + pos % bs;
    req->partial.push_back(token_ids[i]);
    if ((int32_t)req->partial.size() == bs) {  // the block is full: register it
      const Key k = chain(req->last, req->partial.data(), bs);
      if (p->map.find(k) == p->map.end()) {
        p->map.emplace(k, id);
        p->cached[id] = 1;
        p->key[id] = k;
        std::memcpy(&p->toks[(size_t)id * bs], req->partial.data(), sizeof(int32_t) * bs);
      }
      req->last = k;
      req->partial.clear();
    }
  }
  req->ntok = t0 + num_tokens;
  return PKV_OK;
}

int pkv_request_fork(const pkv_request* req, pkv_request** out) {
  if (!out) return PKV_ERR_INVALID_ARG;
  *out = nullptr;
  if (!req) return PKV_ERR_INVALID_ARG;
  pkv_request* c = new (std::nothrow) pkv_request(*req);
  if (!c) return PKV_ERR_INVALID_ARG;
  for (int32_t id : c->table) ++c->pool->ref[id];
  *out = c;
  return PKV_OK;
}

void pkv_request_free(pkv_request* req) {
  if (!req) return;
  for (size_t j = req->table.size(); j-- > 0;) req->pool->release(req->table[j]);
  delete req;
}

int32_t pkv_request_num_tokens(const pkv_request* req) { return req ? req->ntok : -1; }

int32_t pkv_request_block_table(const pkv_request* req, int32_t* out, int32_t max) {
  if (!req) return -1;
  const int32_t n = (int32_t)req->table.size();
  for (int32_t j = 0; j < n && j < max; ++j) out[j] = req->table[j];
  return n;
}

int pkv_requests_block_tables(const pkv_request* const* reqs, int32_t num_reqs,
                              int32_t max_blocks, int32_t* block_tables, int32_t* context_lens) {
  if (num_reqs < 0 || max_blocks <= 0) return PKV_ERR_INVALID_ARG;
  if (num_reqs > 0 && (!reqs || !block_tables)) return PKV_ERR_INVALID_ARG;
  for (int32_t i = 0; i < num_reqs; ++i)
    if (!reqs[i] || (int64_t)reqs[i]->table.size() > max_blocks) return PKV_ERR_INVALID_ARG;
  for (int32_t i = 0; i < num_reqs; ++i) {
    const pkv_request* r = reqs[i];
    int32_t* row = block_tables + (size_t)i * max_blocks;
    const int32_t n = (int32_t)r->table.size();
    if (n > 0) std::memcpy(row, r->table.data(), sizeof(int32_t) * n);
    for (int32_t j = n; j < max_blocks; ++j) row[j] = 0;
    if (context_lens) context_lens[i] = r->ntok;
  }
  return PKV_OK;
}

}  // extern "C"
