"""Prefix cache (host only): the oracle pinned to the published FNV-1a
test vectors and to properties the definition fixes, planted mistakes that
the pins must catch, and the library against the oracle bit for bit over
random token streams and random insert / match / erase sequences.

Definition: "KV-Cache Engineering: Paged Attention, Prefix Cache,
Disaggregation (2026)", prefix caching answer (cumulative hash per block,
hash -> block map, block-by-block walk) and cross-layer sharing answer (per
layer group); "KV Cache Engineering: PagedAttention, Continuous Batching,
Attention Variants, and the Bandwidth Wall", "Prefix Caching" (full blocks).
"""
import os
import random
import types

import pytest

import paged_kv_cache_274_gb300 as pkv
from oracle import prefix_cache as opc


# ---------------------------------------------------------------------------
# pins of the oracle (each takes the oracle module so mutants can run them)
# ---------------------------------------------------------------------------
def pin_fnv_vectors(m):
    # published FNV-1a 64-bit test vectors (Fowler/Noll/Vo test suite)
    assert m.fnv1a64(b"") == 0xCBF29CE484222325
    assert m.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert m.fnv1a64(b"foobar") == 0x85944171F73967E8


def pin_cumulative(m):
    r = random.Random(5)
    a = [r.randrange(50000) for _ in range(16 * 6)]
    b = list(a)
    b[16 * 3 + 7] += 1                       # change one token of block 3
    ha, hb = m.block_hashes(a, 16), m.block_hashes(b, 16)
    assert len(ha) == 6
    assert ha[:3] == hb[:3] and all(x != y for x, y in zip(ha[3:], hb[3:]))
    # the same block content after a different prefix hashes differently
    c = [7] * 16 + a[16:32]
    d = [8] * 16 + a[16:32]
    assert m.block_hashes(c, 16)[1] != m.block_hashes(d, 16)[1]
    # only full blocks: a partial tail adds nothing and changes nothing
    assert m.block_hashes(a + [1, 2, 3], 16) == ha
    assert m.block_hashes(a[:15], 16) == []


def pin_token_bytes(m):
    # 32-bit two's complement, little endian: -1 and 2^32 - 1 are one id,
    # and swapping two tokens changes the hash
    assert m.block_hashes([-1, 5], 2) == m.block_hashes([2**32 - 1, 5], 2)
    assert m.block_hashes([1, 2], 2) != m.block_hashes([2, 1], 2)
    assert m.block_hashes([1, 2], 2) != m.block_hashes([1 << 8, 2], 2)


def pin_byte_layout(m):
    # the hashed bytes, serialised independently with struct: LE64 parent
    # hash (0 for the first block), then LE32 tokens
    import struct
    h0 = m.fnv1a64(struct.pack("<Q", 0) + struct.pack("<3i", 1, -2, 70000))
    h1 = m.fnv1a64(struct.pack("<Q", h0) + struct.pack("<3i", 5, 6, 7))
    assert m.block_hashes([1, -2, 70000, 5, 6, 7], 3) == [h0, h1]


def pin_walk(m):
    bs = 4
    c = m.PrefixCache(bs, 2)
    sys_prompt = list(range(100, 112))                    # 3 full blocks
    req1 = sys_prompt + [1, 2, 3, 4, 5]                   # + 1 full block + tail
    assert c.insert(0, req1, [10, 11, 12, 13, 14]) == 4   # the partial 5th block is not cached
    req2 = sys_prompt + [9, 9, 9, 9, 9, 9]
    assert c.match(0, req2) == [10, 11, 12]               # stops at the first miss
    assert c.match(0, req1) == [10, 11, 12, 13]
    assert c.match(0, req1, max_blocks=2) == [10, 11]
    assert c.match(1, req1) == []                         # groups are separate
    assert c.match(0, [5] + req1[1:]) == []               # first block differs: nothing
    assert c.stats(0) == (4, 3 + 1 + 4 + 2 + 1, 3 + 4 + 2)
    # a second writer of the same prefix keeps the first entries
    assert c.insert(0, req1, [20, 21, 22, 23]) == 0
    assert c.match(0, req1) == [10, 11, 12, 13]
    # erasing a middle block cuts the walk there
    assert c.erase(0, [11, 99]) == 1
    assert c.match(0, req1) == [10]
    # re-registering the prefix into other blocks restores the walk
    assert c.insert(0, req1, [10, 31, 12, 13]) == 1
    assert c.match(0, req1) == [10, 31, 12, 13]
    # a block holds one entry: reusing block 13 for other content drops the old
    assert c.insert(0, [0, 0, 0, 0], [13]) == 1
    assert c.match(0, req1) == [10, 31, 12]


PINS = [pin_fnv_vectors, pin_cumulative, pin_token_bytes, pin_byte_layout, pin_walk]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(opc)


MUTANTS = [
    ("fnv1_order", "        h ^= octet\n        h = (h * FNV64_PRIME) & MASK64",
     "        h = (h * FNV64_PRIME) & MASK64\n        h ^= octet"),
    ("not_cumulative", "data = _le(parent, 8) + ", "data = _le(0, 8) + "),
    ("big_endian_tokens", "return (value & ((1 << (8 * nbytes)) - 1)).to_bytes(nbytes, \"little\")",
     "return (value & ((1 << (8 * nbytes)) - 1)).to_bytes(nbytes, \"big\")"),
    ("partial_block_hashed", "for j in range(len(tokens) // block_size):",
     "for j in range(-(-len(tokens) // block_size)):"),
    ("walk_skips_miss", "                break\n            self.hits", "                continue\n            self.hits"),
    ("no_token_check", "if entry is None or entry[1] != parent or entry[2] != block_tokens:",
     "if entry is None:"),
    ("last_writer_wins", "            if h not in self.maps[group]:", "            if True:"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistakes(name, old, new):
    src = open(opc.__file__).read()
    assert src.count(old) == 1, f"anchor not found: {name}"
    mod = types.ModuleType(f"mutant_{name}")
    exec(compile(src.replace(old, new), f"mutant_{name}.py", "exec"), mod.__dict__)
    failed = []
    for pin in PINS:
        try:
            pin(mod)
        except (AssertionError, KeyError, IndexError):
            failed.append(pin.__name__)
    if name == "no_token_check":
        # a bare hash match cannot be told apart without a collision; force one
        try:
            _collision_pin(mod)
        except AssertionError:
            failed.append("collision")
    assert failed, f"no pin caught the planted mistake {name}"


def _collision_pin(m):
    # an entry whose hash matches but whose tokens differ must not hit
    c = m.PrefixCache(2)
    c.insert(0, [1, 2], [7])
    h = m.block_hashes([1, 2], 2)[0]
    blk, parent, toks = c.maps[0][h]
    c.maps[0][h] = (blk, parent, [3, 4])      # same hash, other content
    assert c.match(0, [1, 2]) == []


def test_collision_guard():
    _collision_pin(opc)


# ---------------------------------------------------------------------------
# library vs oracle
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("bs", [1, 2, 16, 32])
def test_hashes_bit_exact(bs):
    r = random.Random(bs)
    for n in (0, bs - 1, bs, 5 * bs + 3, 64 * bs):
        toks = [r.randrange(-2**31, 2**31) for _ in range(n)]
        assert pkv.prefix_block_hashes(toks, bs) == opc.block_hashes(toks, bs)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_operation_sequences_match_oracle(seed):
    r = random.Random(seed)
    bs, groups = 4, 2
    lib, ref = pkv.PrefixCache(bs, groups), opc.PrefixCache(bs, groups)
    prompts = [[r.randrange(1000) for _ in range(bs * r.randrange(1, 5))] for _ in range(4)]
    next_block = 0
    for _ in range(400):
        g = r.randrange(groups)
        op = r.random()
        toks = r.choice(prompts) + [r.randrange(1000) for _ in range(r.randrange(0, 3 * bs))]
        if op < 0.45:
            assert lib.match(toks, g) == ref.match(g, toks)
        elif op < 0.85:
            nb = len(toks) // bs + r.randrange(0, 2)
            ids = list(range(next_block, next_block + nb))
            if r.random() < 0.3 and next_block > 0:      # reuse some freed ids
                ids = [r.randrange(next_block) for _ in range(nb)]
            next_block += nb
            assert lib.insert(toks, ids, g) == ref.insert(g, toks, ids)
        else:
            ids = [r.randrange(max(1, next_block)) for _ in range(r.randrange(1, 6))]
            assert lib.erase(ids, g) == ref.erase(g, ids)
        assert lib.stats(g) == ref.stats(g)


def test_argument_errors():
    with pytest.raises(pkv.PkvError):
        pkv.PrefixCache(0)
    c = pkv.PrefixCache(4, 1)
    with pytest.raises(pkv.PkvError):
        c.match([1, 2, 3, 4], group=1)
    with pytest.raises(pkv.PkvError):
        c.insert([1, 2, 3, 4], [-1])
    c.close()
