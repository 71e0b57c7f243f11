"""CPU oracle for paged decode attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never imports it and shares no code with it.

The arithmetic lives in ``pkv_oracle.c`` (plain C, float64); this module
compiles it with gcc on first use and wraps it with ctypes.  ``formulas.py``
holds the pages' byte-accounting formulas.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

from .formulas import (  # noqa: F401
    kv_bytes_per_token,
    kv_bytes,
    kv_bytes_per_token_grouped,
    decode_kv_read_seconds,
    blocks_for_tokens,
    last_block_waste_tokens,
    tokens_that_fit,
    naive_utilisation,
)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libpkv_oracle.so")
_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None

ORACLE_OK = 0
ORACLE_BAD_ARG = -1
ORACLE_BAD_BLOCK = -2
ORACLE_BAD_SLOT = -3
ORACLE_BAD_CTX = -4


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc, -O2, OpenMP, no fast-math, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Declare the C signatures on a loaded oracle library."""
    P = ctypes.c_void_p
    i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.pkv_oracle_e4m3_decode.restype = ctypes.c_double
    lib.pkv_oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.pkv_oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.pkv_oracle_e4m3_encode.argtypes = [f32]
    lib.pkv_oracle_e4m3_decode_array.restype = None
    lib.pkv_oracle_e4m3_decode_array.argtypes = [P, P, i64]
    lib.pkv_oracle_e4m3_quantize_array.restype = None
    lib.pkv_oracle_e4m3_quantize_array.argtypes = [P, P, P, i64]
    lib.pkv_oracle_kv_append.restype = ctypes.c_int
    lib.pkv_oracle_kv_append.argtypes = [P, P, P, i32, P, P, i32, P, P,
                                         i32, i32, i32, i32, i32, i32]
    lib.pkv_oracle_paged_decode.restype = ctypes.c_int
    lib.pkv_oracle_paged_decode.argtypes = [P, i32, i32, P, P, i32, P, P,
                                            i32, i32, i32, i32, i32,
                                            P, i32, P, P, i32, i32, f32, P, P, i32]
    lib.pkv_oracle_paged_decode_multi.restype = ctypes.c_int
    lib.pkv_oracle_paged_decode_multi.argtypes = [P, i32, i32, i32, P, P, i32, P, P,
                                                  i32, i32, i32, i32, i32,
                                                  P, i32, P, P, i32, i32, f32, P, P, i32]
    lib.pkv_oracle_int8_encode.restype = ctypes.c_int8
    lib.pkv_oracle_int8_encode.argtypes = [f32, f32, f32]
    lib.pkv_oracle_int8_decode.restype = ctypes.c_double
    lib.pkv_oracle_int8_decode.argtypes = [ctypes.c_int8, f32, f32]
    lib.pkv_oracle_copy_blocks.restype = ctypes.c_int
    lib.pkv_oracle_copy_blocks.argtypes = [P, P, P, P, i32, P, P, P, P, i32, P, i32, i64, i32]
    lib.pkv_oracle_num_threads.restype = ctypes.c_int
    lib.pkv_oracle_num_threads.argtypes = []
    return lib


def load_library(path: str) -> ctypes.CDLL:
    """Load another build of the oracle source (used to plant mistakes in tests)."""
    return _bind(ctypes.CDLL(path))


def _load(lib: Optional[ctypes.CDLL] = None) -> ctypes.CDLL:
    global _lib
    if lib is not None:
        return lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _kind(cache: np.ndarray) -> int:
    """Element kind of a cache array: 0 bf16 bits (uint16), 1 E4M3 codes
    (uint8), 2 INT8 codes (int8)."""
    return {np.dtype(np.uint16): 0, np.dtype(np.uint8): 1, np.dtype(np.int8): 2}[cache.dtype]


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().pkv_oracle_num_threads())


# ---------------------------------------------------------------------------
# E4M3 codec
# ---------------------------------------------------------------------------
def e4m3_decode(codes, lib=None) -> np.ndarray:
    """float64 values of E4M3 codes (any shape)."""
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load(lib).pkv_oracle_e4m3_decode_array(_ptr(c), _ptr(out), c.size)
    return out


def e4m3_encode(x: float, lib=None) -> int:
    return int(_load(lib).pkv_oracle_e4m3_encode(float(np.float32(x))))


def e4m3_quantize(x_bf16_bits, scales_per_elem, lib=None) -> np.ndarray:
    """E4M3 codes of float(x) / scale (binary32 division), elementwise."""
    x = _c(x_bf16_bits, np.uint16)
    s = _c(np.broadcast_to(scales_per_elem, x.shape), np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _load(lib).pkv_oracle_e4m3_quantize_array(_ptr(x), _ptr(s), _ptr(out), x.size)
    return out


def quantize_cache(src_bits: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """E4M3 cache [S][NB][Hkv][bs][D] from bf16 source and [S][NB][Hkv] scales."""
    S, NB, Hkv, bs, D = src_bits.shape
    out = np.empty(src_bits.shape, dtype=np.uint8)
    lib = _load()
    # one page-chunk at a time keeps the broadcast scale array small
    flat_src = src_bits.reshape(S * NB * Hkv, bs * D)
    flat_out = out.reshape(S * NB * Hkv, bs * D)
    flat_sc = scales.reshape(-1)
    step = 1 << 13
    for s in range(0, flat_src.shape[0], step):
        e = min(flat_src.shape[0], s + step)
        x = np.ascontiguousarray(flat_src[s:e])
        sc = np.ascontiguousarray(np.repeat(flat_sc[s:e, None], bs * D, axis=1), dtype=np.float32)
        o = np.empty(x.shape, dtype=np.uint8)
        lib.pkv_oracle_e4m3_quantize_array(_ptr(x), _ptr(sc), _ptr(o), x.size)
        flat_out[s:e] = o
    return out


# ---------------------------------------------------------------------------
# KV append and paged decode
# ---------------------------------------------------------------------------
def kv_append(k_new, v_new, slot_mapping, k_cache: np.ndarray, v_cache: np.ndarray,
              k_scale=None, v_scale=None, slot: int = 0, lib=None) -> int:
    """In-place scatter of new tokens into ``k_cache``/``v_cache`` (numpy).

    Caches are ``[S][NB][Hkv][bs][D]`` uint16 (bf16 bits), uint8 (E4M3) or
    int8 (INT8; scales then [S][NB][Hkv][2] = (scale, zero)).
    Returns the oracle status (0 = ok)."""
    kind = _kind(k_cache)
    fp8 = kind != 0
    S, NB, Hkv, bs, D = k_cache.shape
    kn = _c(k_new, np.uint16)
    vn = _c(v_new, np.uint16)
    sm = _c(slot_mapping, np.int64)
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    ks = _c(k_scale, np.float32) if fp8 else None
    vs = _c(v_scale, np.float32) if fp8 else None
    return int(_load(lib).pkv_oracle_kv_append(
        _ptr(kn), _ptr(vn), _ptr(sm), int(sm.shape[0]), _ptr(k_cache), _ptr(v_cache),
        kind, _ptr(ks), _ptr(vs), S, NB, Hkv, bs, D, int(slot)))


def paged_decode(q_bits, k_cache, v_cache, block_tables, context_lens, kv_group_ptr,
                 layer: int, scale: float, k_scale=None, v_scale=None,
                 pairs=None, lib=None) -> np.ndarray:
    """float64 [B][Hq][D] attention output (see pkv_oracle.c for the definition).

    ``pairs``: optional int array [n][2] of (b, h) to compute; other entries
    of the result are NaN.  Raises ValueError on an oracle status != 0."""
    q = _c(q_bits, np.uint16)
    B, Hq, D = q.shape
    kind = _kind(k_cache)
    fp8 = kind != 0
    kc = _c(k_cache, k_cache.dtype)
    vc = _c(v_cache, v_cache.dtype)
    S, NB, Hkv, bs, Dc = kc.shape
    assert Dc == D
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    gp = _c(kv_group_ptr, np.int32)
    ks = _c(k_scale, np.float32) if fp8 else None
    vs = _c(v_scale, np.float32) if fp8 else None
    out = np.full((B, Hq, D), np.nan if pairs is not None else 0.0, dtype=np.float64)
    pr = None if pairs is None else np.unique(_c(pairs, np.int32).reshape(-1, 2), axis=0)
    rc = _load(lib).pkv_oracle_paged_decode(
        _ptr(q), B, Hq, _ptr(kc), _ptr(vc), kind, _ptr(ks), _ptr(vs),
        S, NB, Hkv, bs, D, _ptr(bt), int(bt.shape[1]), _ptr(cl), _ptr(gp), int(gp.shape[0]),
        int(layer), float(np.float32(scale)), _ptr(out), _ptr(pr),
        0 if pr is None else int(pr.shape[0]))
    if rc != ORACLE_OK:
        raise ValueError(f"oracle paged_decode status {rc}")
    return out


def paged_decode_multi(q_bits, k_cache, v_cache, block_tables, context_lens, kv_group_ptr,
                       layer: int, scale: float, k_scale=None, v_scale=None,
                       rows=None, lib=None) -> np.ndarray:
    """float64 [B][T][Hq][D] output of a T-token query step (query token t of
    sequence b attends to its first context_lens[b] - T + t + 1 cached
    tokens; see pkv_oracle.c).  ``rows``: optional int array [n][3] of
    (b, t, h) to compute; other entries of the result are NaN."""
    q = _c(q_bits, np.uint16)
    B, T, Hq, D = q.shape
    kind = _kind(k_cache)
    fp8 = kind != 0
    kc = _c(k_cache, k_cache.dtype)
    vc = _c(v_cache, v_cache.dtype)
    S, NB, Hkv, bs, Dc = kc.shape
    assert Dc == D
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    gp = _c(kv_group_ptr, np.int32)
    ks = _c(k_scale, np.float32) if fp8 else None
    vs = _c(v_scale, np.float32) if fp8 else None
    out = np.full((B, T, Hq, D), np.nan if rows is not None else 0.0, dtype=np.float64)
    pr = None
    if rows is not None:
        r = np.asarray(rows, dtype=np.int64).reshape(-1, 3)
        pr = np.unique(np.stack([r[:, 0], r[:, 1] * Hq + r[:, 2]], axis=1).astype(np.int32), axis=0)
    rc = _load(lib).pkv_oracle_paged_decode_multi(
        _ptr(q), B, T, Hq, _ptr(kc), _ptr(vc), kind, _ptr(ks), _ptr(vs),
        S, NB, Hkv, bs, D, _ptr(bt), int(bt.shape[1]), _ptr(cl), _ptr(gp), int(gp.shape[0]),
        int(layer), float(np.float32(scale)), _ptr(out), _ptr(pr),
        0 if pr is None else int(pr.shape[0]))
    if rc != ORACLE_OK:
        raise ValueError(f"oracle paged_decode_multi status {rc}")
    return out


def _cache_values(cache: np.ndarray, params, slot: int, blocks: np.ndarray) -> np.ndarray:
    """float64 values of the pages of ``blocks`` in cache slot ``slot``:
    [len(blocks)][Hkv][bs][D].  bf16 bits widen exactly; E4M3 codes take the
    oracle codec's value times the page's fp32 scale; INT8 codes give
    (code - zero) * scale with the page's (scale, zero) -- all exact in
    float64, the same values ``pkv_oracle.c`` reads element by element."""
    pages = cache[slot, blocks]
    kind = _kind(cache)
    if kind == 0:
        return (pages.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if kind == 1:
        table = e4m3_decode(np.arange(256, dtype=np.uint8))
        sc = np.asarray(params, np.float32)[slot, blocks].astype(np.float64)
        return table[pages] * sc[:, :, None, None]
    pr = np.asarray(params, np.float32)[slot, blocks].astype(np.float64)  # [n][Hkv][2]
    return (pages.astype(np.float64) - pr[:, :, None, None, 1]) * pr[:, :, None, None, 0]


def paged_decode_multi_gemm(q_bits, k_cache, v_cache, block_tables, context_lens, kv_group_ptr,
                            layer: int, scale: float, k_scale=None, v_scale=None) -> np.ndarray:
    """float64 [B][T][Hq][D]: the definition of ``paged_decode_multi`` with the
    logits and the weighted sum of values of each (sequence, KV head) taken
    as float64 matrix products over the gathered logical sequence.

    For sequence b with n = context_lens[b] cached tokens (the last T of them
    the new ones) and KV head g ("KV Cache Engineering: PagedAttention,
    Continuous Batching, Attention Variants, and the Bandwidth Wall", "What
    the KV Cache Stores and Why", "PagedAttention", "Attention Variants"):
      K, V  = the n rows of KV head g gathered through block_tables[b] from
              cache slot kv_group_ptr[layer] (dequantised for E4M3 / INT8);
      Q     = the (query token t, head h) rows with h / G == g, [T*G][D];
      S     = double(scale) * Q K^T, with row (t, .) keeping only the keys
              at positions 0 .. n - T + t (causal among the new tokens);
      P     = exp(S - rowmax S) / rowsum exp(S - rowmax S);
      out   = P V  (rows with no position to attend to are zero).
    The matrix products sum in a different order than the element-by-element
    C oracle, so the two agree to float64 rounding (about 1e-15 relative),
    not bit for bit.  Raises ValueError for a context length or a table entry
    outside its range (nothing is read out of bounds)."""
    q = _c(q_bits, np.uint16)
    B, T, Hq, D = q.shape
    S_, NB, Hkv, bs, Dc = k_cache.shape
    assert Dc == D and Hq % Hkv == 0
    G = Hq // Hkv
    bt = np.asarray(block_tables, np.int64)
    cl = np.asarray(context_lens, np.int64)
    slot = int(np.asarray(kv_group_ptr)[layer])
    if not 0 <= slot < S_:
        raise ValueError("kv_group_ptr entry outside the cache slots")
    sc = float(np.float32(scale))
    qf = (q.astype(np.uint32) << 16).view(np.float32).astype(np.float64)  # [B][T][Hq][D]
    out = np.zeros((B, T, Hq, D), dtype=np.float64)
    pos_t = np.arange(T)
    for b in range(B):
        n = int(cl[b])
        if n < 0 or n > bt.shape[1] * bs:
            raise ValueError(f"context_lens[{b}] = {n} out of range")
        if n == 0:
            continue
        blocks = bt[b, :(n + bs - 1) // bs]
        if np.any((blocks < 0) | (blocks >= NB)):
            raise ValueError(f"block_tables[{b}] holds an id outside [0, {NB})")
        # [Hkv][n][D] in logical token order
        K = _cache_values(k_cache, k_scale, slot, blocks).transpose(1, 0, 2, 3).reshape(Hkv, -1, D)[:, :n]
        V = _cache_values(v_cache, v_scale, slot, blocks).transpose(1, 0, 2, 3).reshape(Hkv, -1, D)[:, :n]
        keys = n - T + pos_t + 1                       # keys query token t sees
        visible = np.arange(n)[None, :] < keys[:, None]  # [T][n]
        for g in range(Hkv):
            Q = qf[b, :, g * G:(g + 1) * G, :].reshape(T * G, D)       # rows (t, i)
            S = sc * (Q @ K[g].T)                                       # [T*G][n]
            mask = np.repeat(visible, G, axis=0)
            S = np.where(mask, S, -np.inf)
            smax = S.max(axis=1, keepdims=True)
            live = np.isfinite(smax[:, 0])
            E = np.where(mask, np.exp(S - np.where(live[:, None], smax, 0.0)), 0.0)
            z = E.sum(axis=1, keepdims=True)
            O = (E / np.where(z > 0, z, 1.0)) @ V[g]
            O[~live] = 0.0
            out[b, :, g * G:(g + 1) * G, :] = O.reshape(T, G, D)
    return out


def copy_blocks(src_k, src_v, dst_k, dst_v, pairs, src_k_scale=None, src_v_scale=None,
                dst_k_scale=None, dst_v_scale=None, lib=None) -> int:
    """In-place block copy between pools [NB][Hkv][bs][D] (numpy, any dtype),
    pairs (src, dst) applied in order.  Returns the oracle status."""
    pr = _c(pairs, np.int32).reshape(-1, 2)
    for a in (src_k, src_v, dst_k, dst_v):
        assert a.flags.c_contiguous
    nb_bytes = int(np.prod(src_k.shape[1:])) * src_k.dtype.itemsize
    fp8 = src_k_scale is not None
    hkv = int(src_k.shape[1]) * (2 if src_k.dtype == np.int8 else 1)
    return int(_load(lib).pkv_oracle_copy_blocks(
        _ptr(src_k), _ptr(src_v), _ptr(src_k_scale), _ptr(src_v_scale), int(src_k.shape[0]),
        _ptr(dst_k), _ptr(dst_v), _ptr(dst_k_scale), _ptr(dst_v_scale), int(dst_k.shape[0]),
        _ptr(pr), int(pr.shape[0]), nb_bytes, hkv if fp8 else 0))


def int8_encode(x: float, scale: float, zero: float = 0.0, lib=None) -> int:
    return int(_load(lib).pkv_oracle_int8_encode(float(np.float32(x)), float(np.float32(scale)),
                                                  float(np.float32(zero))))


def int8_decode(q: int, scale: float, zero: float = 0.0, lib=None) -> float:
    return float(_load(lib).pkv_oracle_int8_decode(int(q), float(np.float32(scale)), float(np.float32(zero))))


def int8_quantize_cache(src_bits: np.ndarray, params: np.ndarray) -> np.ndarray:
    """INT8 cache [S][NB][Hkv][bs][D] from bf16 source and [S][NB][Hkv][2]
    (scale, zero) page parameters, through the oracle's append of every row."""
    S, NB, Hkv, bs, D = src_bits.shape
    out = np.zeros(src_bits.shape, dtype=np.int8)
    other = np.zeros(src_bits.shape, dtype=np.int8)
    tok = np.ascontiguousarray(np.transpose(src_bits, (0, 1, 3, 2, 4)))  # [S][NB][bs][Hkv][D]
    for s_ in range(S):
        rows = tok[s_].reshape(NB * bs, Hkv, D)
        slots = np.arange(NB * bs, dtype=np.int64)
        rc = kv_append(rows, rows, slots, out, other, params, params, slot=s_)
        assert rc == 0
    return out
