/*
 * pkv prefix cache -- host-side index of cached KV blocks by content.
 *
 * Sources:
 *   [PC] "KV-Cache Engineering: Paged Attention, Prefix Cache,
 *        Disaggregation (2026)", "How does prefix caching work and what hit
 *        rates are achievable?": a cumulative content hash per block of the
 *        page pool, one global hash -> physical block lookup, and a new
 *        request walks its prefix block by block; matching blocks are reused
 *        (its block table points at the existing physical blocks) and the
 *        first block that does not match is where prefill starts.  Same page,
 *        "What is cross-layer KV sharing ...": the cumulative hash is kept
 *        per layer group.
 *   [BW] "KV Cache Engineering: PagedAttention, Continuous Batching,
 *        Attention Variants, and the Bandwidth Wall", "Prefix Caching" /
 *        "How vLLM implements automatic prefix caching": only full blocks
 *        are hashed, and a hit maps the cached physical block into the new
 *        request's block table.
 *
 * Definitions (the pages name no hash function; this library fixes one):
 *   FNV-1a 64-bit: h = 0xcbf29ce484222325; for each byte c: h = (h ^ c) *
 *     0x100000001b3 mod 2^64.
 *   Block hash: block j of a token sequence (tokens j*bs .. j*bs+bs-1, full
 *     blocks only) has
 *       H_j = FNV-1a-64( LE64(H_{j-1}) || LE32(tok_{j*bs}) || ... || LE32(tok_{j*bs+bs-1}) ),
 *     H_{-1} = 0, token ids taken as 32-bit two's complement, LE = little
 *     endian bytes.  H_j therefore depends on the whole prefix up to the end
 *     of block j ("cumulative").
 *   A lookup of block j hits only if an entry with hash H_j exists in the
 *   group AND its stored tokens equal the block's tokens AND its stored
 *   parent hash equals H_{j-1}: a hash collision can never map a block with
 *   different content (or a different prefix) into a table.
 *
 * All functions are host only (no GPU work, no CUDA calls) and thread safe
 * on one cache object (an internal mutex).  Status codes as in pkv.h.
 */
#ifndef PKV_PREFIX_H_
#define PKV_PREFIX_H_

#include <stddef.h>
#include <stdint.h>

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_prefix_cache pkv_prefix_cache; /* opaque */

/*
 * Hashes of the full blocks of a token sequence (no cache object needed):
 * hashes[j] = H_j for j < num_tokens / block_size.  `hashes` is host memory
 * of at least num_tokens / block_size entries (may be NULL when that is 0).
 */
pkv_status pkv_prefix_block_hashes(int32_t block_size, const int32_t* tokens, int64_t num_tokens,
                                   uint64_t* hashes);

/*
 * A cache with `num_groups` independent layer groups (each with its own
 * hash -> block map; a layout whose block ids serve every group uses one
 * group), for blocks of `block_size` tokens.  *cache is owned by the caller
 * and released with pkv_prefix_cache_destroy.
 */
pkv_status pkv_prefix_cache_create(int32_t block_size, int32_t num_groups, pkv_prefix_cache** cache);
pkv_status pkv_prefix_cache_destroy(pkv_prefix_cache* cache);

/*
 * Walk the full blocks of `tokens` in order and stop at the first block
 * that is not cached in `group`.  block_ids[j] (host, room for max_blocks)
 * receives the physical block of matched block j; *num_matched = matched
 * blocks (at most max_blocks).  Counts one lookup per block tried and one
 * hit per block matched (see pkv_prefix_cache_stats).
 */
pkv_status pkv_prefix_cache_match(pkv_prefix_cache* cache, int32_t group, const int32_t* tokens,
                                  int64_t num_tokens, int32_t* block_ids, int32_t max_blocks,
                                  int32_t* num_matched);

/*
 * Register the full blocks of a sequence whose KV is in physical blocks
 * block_ids[0 .. num_blocks-1] (its block table order).  Only the first
 * min(num_blocks, num_tokens / block_size) blocks are full; a partial last
 * block is never registered.  A block whose hash is already cached keeps
 * the existing entry (first writer wins); a physical block id may hold one
 * entry per group at a time (registering it again under another hash
 * replaces its old entry).  *num_inserted = new entries.
 */
pkv_status pkv_prefix_cache_insert(pkv_prefix_cache* cache, int32_t group, const int32_t* tokens,
                                   int64_t num_tokens, const int32_t* block_ids, int32_t num_blocks,
                                   int32_t* num_inserted);

/*
 * Forget physical blocks (freed or evicted, or about to be overwritten):
 * their entries leave the group's map.  Ids without an entry are ignored.
 * Blocks cached after an erased one stay in the map but are unreachable by
 * a walk until the erased block is registered again.  *num_erased may be
 * NULL.
 */
pkv_status pkv_prefix_cache_erase(pkv_prefix_cache* cache, int32_t group, const int32_t* block_ids,
                                  int32_t count, int32_t* num_erased);

/* Entries in `group`, and lookups / hits counted by match since creation. */
pkv_status pkv_prefix_cache_stats(const pkv_prefix_cache* cache, int32_t group, int64_t* num_entries,
                                  int64_t* lookups, int64_t* hits);

#ifdef __cplusplus
}
#endif

#endif /* PKV_PREFIX_H_ */
