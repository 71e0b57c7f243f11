"""Seeded synthetic decode workloads (no attention arithmetic lives here).

Every builder returns a :class:`DecodeCase` whose arrays are plain numpy:

* bf16 values are carried as ``uint16`` bit patterns (numpy has no bf16);
  they are drawn as float32 N(0, 1) with numpy's PCG64 generator and rounded
  to bf16 with round-to-nearest-even by torch's CPU conversion;
* the paged cache is ``[S][NB][Hkv][bs][D]`` (S cache slots, i.e. layer
  groups; NB physical blocks; bs tokens per block);
* block tables are ``int32 [B][MB]``; entries past a sequence's last block are
  -1 unless poisoned on purpose;
* FP8 cases carry the bf16 *source* values and one fp32 scale per
  (slot, block, KV head) tile; turning them into E4M3 bytes is the codec's
  job, not this module's.

Seeds follow ``1000 * config + role`` with roles q=1, K=2, V=3, block
permutation=4, context lengths=5, prefix-sharing set=6, appended K=7,
appended V=8, append slots=9; layer ``l`` of a multi-layer query adds
``100 * l`` to the q seed.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

BF16_NAN = np.uint16(0x7FC0)


# ---------------------------------------------------------------------------
# bf16 packing helpers
# ---------------------------------------------------------------------------
def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (RNE, torch CPU) and return the bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def normal_bf16_bits(seed: int, shape, chunk: int = 1 << 24) -> np.ndarray:
    """N(0, 1) float32 draws from PCG64(seed), rounded to bf16; returned as bits.

    Large arrays are produced chunk by chunk from one generator stream so the
    result depends only on ``seed`` and ``shape``.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = bf16_bits_from_f32(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


def fp8_tile_scales(src_bits: np.ndarray) -> np.ndarray:
    """Caller-side scale choice for an E4M3 cache: amax(|tile|) / 448 per tile.

    ``src_bits`` is ``[S][NB][Hkv][bs][D]`` bf16 bits; the tile is one
    (slot, block, KV head) page.  A tile of zeros gets scale 1.  The division
    is done in float32.
    """
    S, NB, Hkv = src_bits.shape[:3]
    out = np.empty((S, NB, Hkv), dtype=np.float32)
    flat = src_bits.reshape(S * NB * Hkv, -1)
    o = out.reshape(-1)
    step = 1 << 14
    for s in range(0, flat.shape[0], step):
        f = np.abs(bf16_bits_to_f32(flat[s:s + step]))
        amax = f.max(axis=1).astype(np.float32)
        sc = (amax / np.float32(448.0)).astype(np.float32)
        sc[amax == 0] = np.float32(1.0)
        o[s:s + step] = sc
    return out


def int8_tile_params(src_bits: np.ndarray, symmetric: bool) -> np.ndarray:
    """Caller-side INT8 page parameters, float32 [S][NB][Hkv][2] = (scale, zero).

    Symmetric: scale = amax(|tile|) / 127, zero = 0.  Asymmetric: scale =
    (max - min) / 255 and zero = rint(-128 - min / scale) clamped to
    [-128, 127].  A constant tile gets scale 1.  float32 arithmetic."""
    S, NB, Hkv = src_bits.shape[:3]
    out = np.empty((S * NB * Hkv, 2), dtype=np.float32)
    flat = src_bits.reshape(S * NB * Hkv, -1)
    step = 1 << 14
    for s in range(0, flat.shape[0], step):
        f = bf16_bits_to_f32(flat[s:s + step])
        if symmetric:
            amax = np.abs(f).max(axis=1).astype(np.float32)
            sc = (amax / np.float32(127.0)).astype(np.float32)
            sc[amax == 0] = np.float32(1.0)
            zero = np.zeros_like(sc)
        else:
            lo = f.min(axis=1).astype(np.float32)
            hi = f.max(axis=1).astype(np.float32)
            sc = ((hi - lo) / np.float32(255.0)).astype(np.float32)
            sc[hi == lo] = np.float32(1.0)
            zero = np.clip(np.rint(np.float32(-128.0) - lo / sc), -128, 127).astype(np.float32)
        out[s:s + step, 0] = sc
        out[s:s + step, 1] = zero
    return out.reshape(S, NB, Hkv, 2)


# ---------------------------------------------------------------------------
# case container
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class DecodeCase:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    bs: int
    S: int
    NB: int
    kv_dtype: str                      # "bf16", "fp8", "int8" (symmetric) or "int8a" (asymmetric)
    context_lens: np.ndarray           # int32 [B]
    block_tables: np.ndarray           # int32 [B][MB]
    kv_group_ptr: np.ndarray           # int32 [L]
    scale: float                       # exactly representable in float32
    q: np.ndarray                      # uint16 [L][B][Hq][D]
    k_src: Optional[np.ndarray]        # uint16 [S][NB][Hkv][bs][D] (None: structure only)
    v_src: Optional[np.ndarray]
    k_scale: Optional[np.ndarray] = None   # float32 [S][NB][Hkv] (fp8) or [S][NB][Hkv][2] (int8)
    v_scale: Optional[np.ndarray] = None
    # optional append step: new tokens written before the decode
    k_new: Optional[np.ndarray] = None     # uint16 [N][Hkv][D]
    v_new: Optional[np.ndarray] = None
    slot_mapping: Optional[np.ndarray] = None  # int64 [N]
    append_slot: int = 0                   # cache slot the append writes into
    notes: Dict[str, object] = dataclasses.field(default_factory=dict)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def MB(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def L(self) -> int:
        return int(self.kv_group_ptr.shape[0])

    def used_rows_mask(self) -> np.ndarray:
        """bool [S][NB][bs]: True where some sequence of some layer reads the row."""
        used = np.zeros((self.S, self.NB, self.bs), dtype=bool)
        for slot in sorted(set(int(x) for x in self.kv_group_ptr)):
            for b in range(self.B):
                n = int(self.context_lens[b])
                for j in range((n + self.bs - 1) // self.bs):
                    rows = min(self.bs, n - j * self.bs)
                    used[slot, self.block_tables[b, j], :rows] = True
        return used


def _scale_for(D: int) -> float:
    return float(np.float32(1.0 / math.sqrt(D)))


def _perm(seed: int, n: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.permutation(n).astype(np.int64)


def _tables_from_counts(nblocks: Sequence[int], phys: np.ndarray, MB: int) -> np.ndarray:
    """Consecutive slices of ``phys`` become the sequences' tables."""
    t = np.full((len(nblocks), MB), -1, dtype=np.int32)
    pos = 0
    for b, n in enumerate(nblocks):
        t[b, :n] = phys[pos:pos + n]
        pos += n
    return t


def _queries(cfg: int, L: int, B: int, Hq: int, D: int) -> np.ndarray:
    return np.stack([normal_bf16_bits(1000 * cfg + 1 + 100 * l, (B, Hq, D)) for l in range(L)])


def _cache(cfg: int, S: int, NB: int, Hkv: int, bs: int, D: int, fill: bool):
    shape = (S, NB, Hkv, bs, D)
    if not fill:   # structure only (block tables, lengths, queries)
        return None, None
    return normal_bf16_bits(1000 * cfg + 2, shape), normal_bf16_bits(1000 * cfg + 3, shape)


def _finish_fp8(case: DecodeCase) -> DecodeCase:
    """Page parameters for one-byte caches: "fp8" (E4M3 scales), "int8"
    (symmetric INT8) and "int8a" (asymmetric INT8)."""
    if case.kv_dtype == "fp8":
        case.k_scale = fp8_tile_scales(case.k_src)
        case.v_scale = fp8_tile_scales(case.v_src)
    elif case.kv_dtype in ("int8", "int8a"):
        sym = case.kv_dtype == "int8"
        case.k_scale = int8_tile_params(case.k_src, sym)
        case.v_scale = int8_tile_params(case.v_src, sym)
    return case


# ---------------------------------------------------------------------------
# the five workloads
# ---------------------------------------------------------------------------
def tiny_case() -> DecodeCase:
    """Tiny paged decode: B 2, 8 q / 2 KV heads, D 64, bs 16, ctx {37, 100},
    the 10 used blocks drawn from a seeded permutation of a 32-block pool."""
    cfg, B, Hq, Hkv, D, bs, NB = 1, 2, 8, 2, 64, 16, 32
    ctx = np.array([37, 100], dtype=np.int32)
    nblk = [(int(c) + bs - 1) // bs for c in ctx]
    phys = _perm(1000 * cfg + 4, NB)
    tables = _tables_from_counts(nblk, phys, max(nblk))
    k, v = _cache(cfg, 1, NB, Hkv, bs, D, True)
    return DecodeCase("tiny", B, Hq, Hkv, D, bs, 1, NB, "bf16", ctx, tables,
                      np.zeros(1, np.int32), _scale_for(D), _queries(cfg, 1, B, Hq, D), k, v)


def llama8b_layer_case(fill: bool = True, B: int = 64, ctx_len: int = 4096) -> DecodeCase:
    """Llama-3.1-8B-shaped decode layer: 32 q / 8 KV heads, D 128, bs 16,
    every context 4096, pool = ceil(1.1 x used blocks); the step first appends
    each sequence's newest token (position ctx-1) into its slot."""
    cfg, Hq, Hkv, D, bs = 2, 32, 8, 128, 16
    per_seq = ctx_len // bs
    used = B * per_seq
    NB = int(math.ceil(1.1 * used - 1e-9))
    phys = _perm(1000 * cfg + 4, NB)[:used]
    tables = _tables_from_counts([per_seq] * B, phys, per_seq)
    ctx = np.full(B, ctx_len, dtype=np.int32)
    k, v = _cache(cfg, 1, NB, Hkv, bs, D, fill)
    last = ctx_len - 1
    slots = np.array([int(tables[b, last // bs]) * bs + last % bs for b in range(B)], dtype=np.int64)
    c = DecodeCase("llama8b_layer", B, Hq, Hkv, D, bs, 1, NB, "bf16", ctx, tables,
                   np.zeros(1, np.int32), _scale_for(D), _queries(cfg, 1, B, Hq, D), k, v,
                   k_new=normal_bf16_bits(1000 * cfg + 7, (B, Hkv, D)),
                   v_new=normal_bf16_bits(1000 * cfg + 8, (B, Hkv, D)),
                   slot_mapping=slots)
    return c


def mixed_prefix_case(fill: bool = True, B: int = 256, lo: int = 128, hi: int = 8192,
                      prefix_tokens: int = 2048) -> DecodeCase:
    """Mixed-length prefix-shared batch: context lengths log-uniform in
    [lo, hi]; a seeded half of the sequences alias the first
    min(ceil(ctx/bs), prefix blocks) table entries to one shared prefix."""
    cfg, Hq, Hkv, D, bs = 3, 32, 8, 128, 16
    rng = np.random.Generator(np.random.PCG64(1000 * cfg + 5))
    ctx = np.rint(np.exp(rng.uniform(math.log(lo), math.log(hi), size=B))).astype(np.int32)
    rng_s = np.random.Generator(np.random.PCG64(1000 * cfg + 6))
    shared = np.zeros(B, dtype=bool)
    shared[rng_s.choice(B, size=B // 2, replace=False)] = True
    pre_blocks = prefix_tokens // bs
    nblk = [(int(c) + bs - 1) // bs for c in ctx]
    # allocation order: prefix blocks, then each sequence's private blocks
    n_private = [n - min(n, pre_blocks) if shared[b] else n for b, n in enumerate(nblk)]
    NB = pre_blocks + sum(n_private)
    phys = _perm(1000 * cfg + 4, NB)
    MB = max(nblk)
    tables = np.full((B, MB), -1, dtype=np.int32)
    pos = pre_blocks
    for b in range(B):
        j0 = 0
        if shared[b]:
            j0 = min(nblk[b], pre_blocks)
            tables[b, :j0] = phys[:j0]
        n = nblk[b] - j0
        tables[b, j0:nblk[b]] = phys[pos:pos + n]
        pos += n
    k, v = _cache(cfg, 1, NB, Hkv, bs, D, fill)
    c = DecodeCase("mixed_prefix", B, Hq, Hkv, D, bs, 1, NB, "bf16", ctx, tables,
                   np.zeros(1, np.int32), _scale_for(D), _queries(cfg, 1, B, Hq, D), k, v)
    c.notes["shared"] = shared
    c.notes["prefix_blocks"] = phys[:pre_blocks].copy()
    return c


def unalias_prefix(case: DecodeCase) -> DecodeCase:
    """Give every sharing sequence private copies of the shared prefix blocks.

    The logical content of every sequence is unchanged; only the physical
    placement differs (new blocks appended to the pool)."""
    shared = case.notes["shared"]
    pre = case.notes["prefix_blocks"]
    extra = []
    tables = case.block_tables.copy()
    nb = case.NB
    for b in range(case.B):
        if not shared[b]:
            continue
        n = (int(case.context_lens[b]) + case.bs - 1) // case.bs
        for j in range(min(n, len(pre))):
            extra.append(int(tables[b, j]))
            tables[b, j] = nb
            nb += 1
    idx = np.array(extra, dtype=np.int64)
    k = np.concatenate([case.k_src, case.k_src[:, idx]], axis=1)
    v = np.concatenate([case.v_src, case.v_src[:, idx]], axis=1)
    c = dataclasses.replace(case, name=case.name + "_private", NB=nb, block_tables=tables,
                            k_src=k, v_src=v, notes=dict(case.notes))
    return c


def long_context_case(variant: str = "b4_32k", fill: bool = True) -> DecodeCase:
    """70B-shaped long context: 64 q / 8 KV heads, D 128, bs 32; batch 4 at
    32768 tokens ("b4_32k") or batch 1 at 131072 tokens ("b1_128k"); the pool
    is exactly the used blocks in a seeded random order."""
    cfg, Hq, Hkv, D, bs = 4, 64, 8, 128, 32
    B, ctx_len = {"b4_32k": (4, 32768), "b1_128k": (1, 131072)}[variant]
    per_seq = ctx_len // bs
    NB = B * per_seq
    seed_off = 0 if variant == "b4_32k" else 10
    phys = _perm(1000 * cfg + 4 + seed_off, NB)
    tables = _tables_from_counts([per_seq] * B, phys, per_seq)
    ctx = np.full(B, ctx_len, dtype=np.int32)
    k, v = _cache(cfg, 1, NB, Hkv, bs, D, fill)
    return DecodeCase("long_" + variant, B, Hq, Hkv, D, bs, 1, NB, "bf16", ctx, tables,
                      np.zeros(1, np.int32), _scale_for(D), _queries(cfg, 1, B, Hq, D), k, v)


def fp8_shared_case(fill: bool = True, B: int = 128, ctx_len: int = 8192, L: int = 4,
                    kv_dtype: str = "fp8") -> DecodeCase:
    """FP8 KV cache with cross-layer sharing: L layers whose shared-with
    pointers all name cache slot 0; B 128, 32 q / 8 KV heads, D 128, bs 32,
    context 8192; per-(block, KV head) fp32 scales from the bf16 N(0,1) data.
    kv_dtype "int8" / "int8a" gives the same workload with an INT8 cache."""
    cfg, Hq, Hkv, D, bs = 5, 32, 8, 128, 32
    per_seq = ctx_len // bs
    NB = B * per_seq
    phys = _perm(1000 * cfg + 4, NB)
    tables = _tables_from_counts([per_seq] * B, phys, per_seq)
    ctx = np.full(B, ctx_len, dtype=np.int32)
    k, v = _cache(cfg, 1, NB, Hkv, bs, D, fill)
    c = DecodeCase(kv_dtype + "_shared", B, Hq, Hkv, D, bs, 1, NB, kv_dtype, ctx, tables,
                   np.zeros(L, np.int32), _scale_for(D), _queries(cfg, L, B, Hq, D), k, v)
    return _finish_fp8(c) if fill else c


CONFIG_BUILDERS = {
    1: tiny_case,
    2: llama8b_layer_case,
    3: mixed_prefix_case,
    4: long_context_case,
    5: fp8_shared_case,
}


# ---------------------------------------------------------------------------
# small random cases for parity sweeps
# ---------------------------------------------------------------------------
def random_case(seed: int, B: int, Hq: int, Hkv: int, D: int, bs: int,
                context_lens: Sequence[int], kv_dtype: str = "bf16", spare_blocks: int = 5,
                S: int = 1, kv_group_ptr: Optional[Sequence[int]] = None,
                poison: bool = False, MB: Optional[int] = None,
                value_scale: float = 1.0) -> DecodeCase:
    """A small seeded case with a random block permutation.

    ``poison`` fills every cache row no sequence reads with bf16 NaN and every
    unused table entry with an out-of-range block id, so that a kernel that
    reads past a sequence's context shows it.  ``value_scale`` multiplies the
    N(0,1) K/V/q draws (to sweep logit ranges)."""
    ctx = np.array(list(context_lens), dtype=np.int32)
    nblk = [(int(c) + bs - 1) // bs for c in ctx]
    need = sum(nblk)
    NB = max(1, need + spare_blocks)
    phys = _perm(seed * 7 + 4, NB)
    mb = MB if MB is not None else max(1, max(nblk) if nblk else 1)
    tables = _tables_from_counts(nblk, phys, mb)
    if poison:
        for b in range(len(ctx)):
            tables[b, nblk[b]:] = NB + 7 + b
    gp = np.array(list(kv_group_ptr) if kv_group_ptr is not None else [0], dtype=np.int32)
    L = len(gp)
    shape = (S, NB, Hkv, bs, D)

    def draw(s, shp):
        if value_scale == 1.0:
            return normal_bf16_bits(s, shp)
        rng = np.random.Generator(np.random.PCG64(s))
        return bf16_bits_from_f32(rng.standard_normal(int(np.prod(shp)), dtype=np.float32)
                                  .reshape(shp) * np.float32(value_scale))

    k = draw(seed * 7 + 2, shape)
    v = draw(seed * 7 + 3, shape)
    q = np.stack([draw(seed * 7 + 1 + 100 * l, (len(ctx), Hq, D)) for l in range(L)])
    c = DecodeCase(f"random{seed}", len(ctx), Hq, Hkv, D, bs, S, NB, kv_dtype, ctx, tables,
                   gp, _scale_for(D), q, k, v)
    c = _finish_fp8(c)
    if poison:
        unused = ~c.used_rows_mask()[:, :, None, :, None]
        c.k_src = np.where(unused, BF16_NAN, c.k_src).astype(np.uint16)
        c.v_src = np.where(unused, BF16_NAN, c.v_src).astype(np.uint16)
        c.notes["poisoned"] = True
    return c
