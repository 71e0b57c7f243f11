// Prefix cache: cumulative FNV-1a-64 block hashes and a per-layer-group
// hash -> physical block index (host only).
//
// Source: "KV-Cache Engineering: Paged Attention, Prefix Cache,
// Disaggregation (2026)", "How does prefix caching work and what hit rates
// are achievable?" (cumulative content hash per block, global hash -> block
// lookup, block-by-block prefix walk that stops at the first miss) and its
// cross-layer sharing answer (the hash is kept per layer group); "KV Cache
// Engineering: PagedAttention, Continuous Batching, Attention Variants, and
// the Bandwidth Wall", "Prefix Caching" (full blocks only).
//
// Each entry keeps the block's tokens and its parent hash, so a lookup hits
// only on identical content after an identical prefix, never on a bare hash
// collision.
#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv_internal.h"
#include "pkv_prefix.h"

namespace {

constexpr uint64_t kFnvOffset = 0xcbf29ce484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001b3ull;

inline uint64_t fnv_byte(uint64_t h, uint8_t c) { return (h ^ c) * kFnvPrime; }

// H_j from H_{j-1} and the block's tokens (little-endian bytes; no reliance
// on the host's byte order).
uint64_t block_hash(uint64_t parent, const int32_t* tok, int bs) {
  uint64_t h = kFnvOffset;
  for (int i = 0; i < 8; ++i) h = fnv_byte(h, static_cast<uint8_t>(parent >> (8 * i)));
  for (int t = 0; t < bs; ++t) {
    const uint32_t u = static_cast<uint32_t>(tok[t]);
    for (int i = 0; i < 4; ++i) h = fnv_byte(h, static_cast<uint8_t>(u >> (8 * i)));
  }
  return h;
}

struct Entry {
  int32_t block;
  uint64_t parent;
  std::vector<int32_t> tokens;
};

struct Group {
  std::unordered_map<uint64_t, Entry> by_hash;
  std::unordered_map<int32_t, uint64_t> hash_of_block;
  int64_t lookups = 0;
  int64_t hits = 0;
};

pkv_status fail(pkv_status st, const char* msg) {
  pkv::set_last_error_message(msg);
  return st;
}

}  // namespace

struct pkv_prefix_cache {
  int32_t bs;
  std::vector<Group> groups;
  mutable std::mutex mu;
};

extern "C" {

pkv_status pkv_prefix_block_hashes(int32_t block_size, const int32_t* tokens, int64_t num_tokens,
                                   uint64_t* hashes) {
  if (block_size < 1 || num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "block_size < 1 or num_tokens < 0");
  const int64_t nb = num_tokens / block_size;
  if (nb > 0 && (tokens == nullptr || hashes == nullptr)) return fail(PKV_ERR_INVALID_ARG, "NULL pointer");
  uint64_t h = 0;
  for (int64_t j = 0; j < nb; ++j) {
    h = block_hash(h, tokens + j * block_size, block_size);
    hashes[j] = h;
  }
  return PKV_OK;
}

pkv_status pkv_prefix_cache_create(int32_t block_size, int32_t num_groups, pkv_prefix_cache** cache) {
  if (cache == nullptr) return fail(PKV_ERR_INVALID_ARG, "cache is NULL");
  *cache = nullptr;
  if (block_size < 1 || num_groups < 1) return fail(PKV_ERR_INVALID_ARG, "block_size and num_groups must be >= 1");
  pkv_prefix_cache* c = new (std::nothrow) pkv_prefix_cache;
  if (c == nullptr) return fail(PKV_ERR_INVALID_ARG, "out of host memory");
  c->bs = block_size;
  c->groups.resize(static_cast<size_t>(num_groups));
  *cache = c;
  return PKV_OK;
}

pkv_status pkv_prefix_cache_destroy(pkv_prefix_cache* cache) {
  delete cache;
  return PKV_OK;
}

static pkv_status check_group(const pkv_prefix_cache* c, int32_t group) {
  if (c == nullptr) return fail(PKV_ERR_INVALID_ARG, "cache is NULL");
  if (group < 0 || static_cast<size_t>(group) >= c->groups.size())
    return fail(PKV_ERR_INVALID_ARG, "group outside [0, num_groups)");
  return PKV_OK;
}

pkv_status pkv_prefix_cache_match(pkv_prefix_cache* cache, int32_t group, const int32_t* tokens,
                                  int64_t num_tokens, int32_t* block_ids, int32_t max_blocks,
                                  int32_t* num_matched) {
  pkv_status st = check_group(cache, group);
  if (st != PKV_OK) return st;
  if (num_matched == nullptr || num_tokens < 0 || max_blocks < 0)
    return fail(PKV_ERR_INVALID_ARG, "num_matched is NULL or a negative size");
  *num_matched = 0;
  const int bs = cache->bs;
  const int64_t nb = std::min<int64_t>(num_tokens / bs, max_blocks);
  if (nb > 0 && (tokens == nullptr || block_ids == nullptr)) return fail(PKV_ERR_INVALID_ARG, "NULL pointer");
  std::lock_guard<std::mutex> lock(cache->mu);
  Group& g = cache->groups[static_cast<size_t>(group)];
  uint64_t parent = 0;
  for (int64_t j = 0; j < nb; ++j) {
    const int32_t* tok = tokens + j * bs;
    const uint64_t h = block_hash(parent, tok, bs);
    ++g.lookups;
    auto it = g.by_hash.find(h);
    if (it == g.by_hash.end() || it->second.parent != parent ||
        std::memcmp(it->second.tokens.data(), tok, sizeof(int32_t) * bs) != 0)
      break;
    ++g.hits;
    block_ids[j] = it->second.block;
    *num_matched = static_cast<int32_t>(j + 1);
    parent = h;
  }
  return PKV_OK;
}

pkv_status pkv_prefix_cache_insert(pkv_prefix_cache* cache, int32_t group, const int32_t* tokens,
                                   int64_t num_tokens, const int32_t* block_ids, int32_t num_blocks,
                                   int32_t* num_inserted) {
  pkv_status st = check_group(cache, group);
  if (st != PKV_OK) return st;
  if (num_tokens < 0 || num_blocks < 0) return fail(PKV_ERR_INVALID_ARG, "negative size");
  const int bs = cache->bs;
  const int64_t nb = std::min<int64_t>(num_tokens / bs, num_blocks);
  if (nb > 0 && (tokens == nullptr || block_ids == nullptr)) return fail(PKV_ERR_INVALID_ARG, "NULL pointer");
  for (int64_t j = 0; j < nb; ++j)
    if (block_ids[j] < 0) return fail(PKV_ERR_INVALID_ARG, "negative block id");
  int32_t added = 0;
  std::lock_guard<std::mutex> lock(cache->mu);
  Group& g = cache->groups[static_cast<size_t>(group)];
  uint64_t parent = 0;
  for (int64_t j = 0; j < nb; ++j) {
    const int32_t* tok = tokens + j * bs;
    const uint64_t h = block_hash(parent, tok, bs);
    if (g.by_hash.find(h) == g.by_hash.end()) {
      const int32_t blk = block_ids[j];
      // a physical block holds one entry: drop what it held before
      auto old = g.hash_of_block.find(blk);
      if (old != g.hash_of_block.end()) g.by_hash.erase(old->second);
      g.by_hash.emplace(h, Entry{blk, parent, std::vector<int32_t>(tok, tok + bs)});
      g.hash_of_block[blk] = h;
      ++added;
    }
    parent = h;
  }
  if (num_inserted != nullptr) *num_inserted = added;
  return PKV_OK;
}

pkv_status pkv_prefix_cache_erase(pkv_prefix_cache* cache, int32_t group, const int32_t* block_ids,
                                  int32_t count, int32_t* num_erased) {
  pkv_status st = check_group(cache, group);
  if (st != PKV_OK) return st;
  if (count < 0 || (count > 0 && block_ids == nullptr)) return fail(PKV_ERR_INVALID_ARG, "bad block list");
  int32_t n = 0;
  std::lock_guard<std::mutex> lock(cache->mu);
  Group& g = cache->groups[static_cast<size_t>(group)];
  for (int32_t i = 0; i < count; ++i) {
    auto it = g.hash_of_block.find(block_ids[i]);
    if (it == g.hash_of_block.end()) continue;
    g.by_hash.erase(it->second);
    g.hash_of_block.erase(it);
    ++n;
  }
  if (num_erased != nullptr) *num_erased = n;
  return PKV_OK;
}

pkv_status pkv_prefix_cache_stats(const pkv_prefix_cache* cache, int32_t group, int64_t* num_entries,
                                  int64_t* lookups, int64_t* hits) {
  pkv_status st = check_group(cache, group);
  if (st != PKV_OK) return st;
  std::lock_guard<std::mutex> lock(cache->mu);
  const Group& g = cache->groups[static_cast<size_t>(group)];
  if (num_entries) *num_entries = static_cast<int64_t>(g.by_hash.size());
  if (lookups) *lookups = g.lookups;
  if (hits) *hits = g.hits;
  return PKV_OK;
}

}  // extern "C"
