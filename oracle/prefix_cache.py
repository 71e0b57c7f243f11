"""Prefix-cache oracle (test infrastructure only: tests/ and bench.py's
reference leg may import it; the product path never does).

Plain-Python restatement of the prefix cache:
"KV-Cache Engineering: Paged Attention, Prefix Cache, Disaggregation (2026)",
"How does prefix caching work and what hit rates are achievable?" -- each
block of the pool gets a cumulative content hash, one map goes from hash to
physical block, and a new request walks its prefix block by block until the
first block that is not cached; the cross-layer sharing answer on the same
page keeps that hash per layer group.  "KV Cache Engineering: PagedAttention,
Continuous Batching, Attention Variants, and the Bandwidth Wall", "Prefix
Caching": only full blocks are hashed.

The pages name no hash function.  The reading taken here (and in the
library): FNV-1a 64-bit (Fowler, Noll, Vo) over the little-endian bytes of
the parent block's hash (8 bytes; 0 before the first block) followed by the
block's token ids as 32-bit two's complement (4 bytes each).
"""
from __future__ import annotations

FNV64_OFFSET = 0xCBF29CE484222325
FNV64_PRIME = 0x100000001B3
MASK64 = (1 << 64) - 1


def fnv1a64(data: bytes) -> int:
    """FNV-1a, 64-bit: for each octet, XOR it into the hash, then multiply
    by the FNV prime modulo 2^64."""
    h = FNV64_OFFSET
    for octet in data:
        h ^= octet
        h = (h * FNV64_PRIME) & MASK64
    return h


def _le(value: int, nbytes: int) -> bytes:
    return (value & ((1 << (8 * nbytes)) - 1)).to_bytes(nbytes, "little")


def block_hashes(tokens, block_size: int) -> list[int]:
    """H_j for every full block j of the token sequence (cumulative: H_j
    hashes H_{j-1} followed by block j's tokens)."""
    out = []
    parent = 0
    for j in range(len(tokens) // block_size):
        data = _le(parent, 8) + b"".join(_le(int(t), 4) for t in tokens[j * block_size:(j + 1) * block_size])
        parent = fnv1a64(data)
        out.append(parent)
    return out


class PrefixCache:
    """hash -> (physical block, parent hash, tokens) per layer group."""

    def __init__(self, block_size: int, num_groups: int = 1):
        self.bs = block_size
        self.maps = [dict() for _ in range(num_groups)]       # hash -> (block, parent, tokens)
        self.block_hash = [dict() for _ in range(num_groups)]  # block -> hash
        self.lookups = [0] * num_groups
        self.hits = [0] * num_groups

    def match(self, group: int, tokens, max_blocks: int | None = None) -> list[int]:
        """Physical blocks of the longest run of leading full blocks that are
        cached with the same tokens after the same prefix."""
        nb = len(tokens) // self.bs
        if max_blocks is not None:
            nb = min(nb, max_blocks)
        found = []
        parent = 0
        hashes = block_hashes(list(tokens[:nb * self.bs]), self.bs)
        for j in range(nb):
            self.lookups[group] += 1
            entry = self.maps[group].get(hashes[j])
            block_tokens = [int(t) for t in tokens[j * self.bs:(j + 1) * self.bs]]
            if entry is None or entry[1] != parent or entry[2] != block_tokens:
                break
            self.hits[group] += 1
            found.append(entry[0])
            parent = hashes[j]
        return found

    def insert(self, group: int, tokens, block_ids) -> int:
        """Register the sequence's full blocks; an already cached hash keeps
        its entry; a physical block holds one entry at a time."""
        nb = min(len(tokens) // self.bs, len(block_ids))
        hashes = block_hashes(list(tokens[:nb * self.bs]), self.bs)
        added = 0
        parent = 0
        for j in range(nb):
            h = hashes[j]
            if h not in self.maps[group]:
                blk = int(block_ids[j])
                if blk in self.block_hash[group]:
                    del self.maps[group][self.block_hash[group][blk]]
                self.maps[group][h] = (blk, parent, [int(t) for t in tokens[j * self.bs:(j + 1) * self.bs]])
                self.block_hash[group][blk] = h
                added += 1
            parent = h
        return added

    def erase(self, group: int, block_ids) -> int:
        n = 0
        for blk in block_ids:
            h = self.block_hash[group].pop(int(blk), None)
            if h is not None:
                del self.maps[group][h]
                n += 1
        return n

    def stats(self, group: int):
        return len(self.maps[group]), self.lookups[group], self.hits[group]
