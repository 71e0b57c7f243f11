"""Paged KV-cache decode attention for GB300 (sm_103a): Python binding.

A thin ctypes layer over the C ABI in ``include/pkv.h`` (library
``_lib/libpkv.so``, built in-tree by ``_build.py``).  It only marshals
arguments: torch tensors supply device pointers and the current CUDA
stream; every step of the computation runs in the library's kernels.  There
is no CPU fallback: if the library is missing or the call fails, a
:class:`PkvError` is raised.

Layouts (see the header for the full contract):
  k_cache, v_cache  [S][NB][Hkv][bs][D]  torch.bfloat16, or torch.uint8 holding
                    E4M3 codes (FP8 cache);
  k_scale, v_scale  float32 [S][NB][Hkv] (FP8 cache only);
  q, out            bfloat16 [B][Hq][D];
  block_tables      int32 [B][MB];  context_lens int32 [B];
  kv_group_ptr      host int32 [L] (shared-with pointer per layer).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libpkv.so")

PKV_OK = 0
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "alignment", 4: "cuda",
                5: "device index error", 6: "workspace"}
KV_BF16, KV_FP8_E4M3, KV_INT8 = 0, 1, 2
MATH_AUTO, MATH_FFMA, MATH_MMA, MATH_TC = 0, 1, 2, 3
DEVERR_BLOCK_ID, DEVERR_SLOT, DEVERR_CONTEXT_LEN, DEVERR_TIMEOUT = 1, 2, 4, 8


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"pkv status {status} ({STATUS_NAMES.get(status, '?')}): {message}")
        self.status = status


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_slots", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class DecodeOpts(ctypes.Structure):
    _fields_ = [("partition_blocks", ctypes.c_int32), ("math", ctypes.c_int32),
                ("warps_per_cta", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("event_decode_start", ctypes.c_void_p), ("event_decode_end", ctypes.c_void_p)]


class DecodePlan(ctypes.Structure):
    _fields_ = [("partition_blocks", ctypes.c_int32), ("max_partitions", ctypes.c_int32),
                ("math", ctypes.c_int32), ("warps_per_cta", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("kernels_per_call", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_size_t), ("smem_bytes_per_cta", ctypes.c_size_t),
                ("query_tokens_per_tile", ctypes.c_int32), ("row_tiles", ctypes.c_int32)]

MAX_QUERY_TOKENS = 512
ABI_VERSION = 2


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return LIB_PATH


def load() -> ctypes.CDLL:
    """Load the built library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise PkvError(4, f"CUDA library not built: {LIB_PATH} is missing "
                              "(run paged_kv_cache_274_gb300._build.build())")
        lib = ctypes.CDLL(LIB_PATH)
        P, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
        pdesc, popts = ctypes.POINTER(CacheDesc), ctypes.POINTER(DecodeOpts)
        lib.pkv_kv_append.restype = ctypes.c_int
        lib.pkv_kv_append.argtypes = [pdesc, i32, P, P, P, i32, P, P, P, P, P]
        lib.pkv_decode_workspace_bytes.restype = sz
        lib.pkv_decode_workspace_bytes.argtypes = [pdesc, i32, i32, i32, popts]
        lib.pkv_decode_describe.restype = ctypes.c_int
        lib.pkv_decode_describe.argtypes = [pdesc, i32, i32, i32, popts, ctypes.POINTER(DecodePlan)]
        lib.pkv_paged_decode.restype = ctypes.c_int
        lib.pkv_paged_decode.argtypes = [pdesc, P, i32, i32, P, P, P, P, P, i32, P, P, i32, i32,
                                         f32, P, P, sz, popts, P]
        lib.pkv_decode_multi_workspace_bytes.restype = sz
        lib.pkv_decode_multi_workspace_bytes.argtypes = [pdesc, i32, i32, i32, i32, popts]
        lib.pkv_decode_multi_describe.restype = ctypes.c_int
        lib.pkv_decode_multi_describe.argtypes = [pdesc, i32, i32, i32, i32, popts,
                                                  ctypes.POINTER(DecodePlan)]
        lib.pkv_paged_decode_multi.restype = ctypes.c_int
        lib.pkv_paged_decode_multi.argtypes = [pdesc, P, i32, i32, i32, P, P, P, P, P, i32, P, P, i32,
                                               i32, f32, P, P, sz, popts, P]
        lib.pkv_append_and_decode.restype = ctypes.c_int
        lib.pkv_append_and_decode.argtypes = [pdesc, P, P, P, i32, P, i32, i32, i32, P, P, P, P, P, i32, P,
                                              P, i32, i32, f32, P, P, sz, popts, P]
        lib.pkv_paged_decode_static_workspace.restype = ctypes.c_int
        lib.pkv_paged_decode_static_workspace.argtypes = [pdesc, P, i32, i32, P, P, P, P, P, i32, P,
                                                          P, i32, i32, f32, P, popts, P]
        lib.pkv_copy_blocks.restype = ctypes.c_int
        lib.pkv_copy_blocks.argtypes = [pdesc, P, P, P, P, i32, P, P, P, P, i32, P, i32, P]
        lib.pkv_read_probe.restype = ctypes.c_int
        lib.pkv_read_probe.argtypes = [P, sz, P, P]
        lib.pkv_read_device_error.restype = ctypes.c_int
        lib.pkv_read_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), P]
        lib.pkv_status_string.restype = ctypes.c_char_p
        lib.pkv_status_string.argtypes = [ctypes.c_int]
        lib.pkv_last_error_message.restype = ctypes.c_char_p
        lib.pkv_last_error_message.argtypes = []
        lib.pkv_abi_version.restype = ctypes.c_int32
        lib.pkv_abi_version.argtypes = []
        i64 = ctypes.c_int64
        pi32 = ctypes.POINTER(ctypes.c_int32)
        pi64 = ctypes.POINTER(ctypes.c_int64)
        lib.pkv_prefix_block_hashes.restype = ctypes.c_int
        lib.pkv_prefix_block_hashes.argtypes = [i32, P, i64, P]
        lib.pkv_prefix_cache_create.restype = ctypes.c_int
        lib.pkv_prefix_cache_create.argtypes = [i32, i32, ctypes.POINTER(ctypes.c_void_p)]
        lib.pkv_prefix_cache_destroy.restype = ctypes.c_int
        lib.pkv_prefix_cache_destroy.argtypes = [P]
        lib.pkv_prefix_cache_match.restype = ctypes.c_int
        lib.pkv_prefix_cache_match.argtypes = [P, i32, P, i64, P, i32, pi32]
        lib.pkv_prefix_cache_insert.restype = ctypes.c_int
        lib.pkv_prefix_cache_insert.argtypes = [P, i32, P, i64, P, i32, pi32]
        lib.pkv_prefix_cache_erase.restype = ctypes.c_int
        lib.pkv_prefix_cache_erase.argtypes = [P, i32, P, i32, pi32]
        lib.pkv_prefix_cache_stats.restype = ctypes.c_int
        lib.pkv_prefix_cache_stats.argtypes = [P, i32, pi64, pi64, pi64]
        if lib.pkv_abi_version() != ABI_VERSION:
            raise RuntimeError(f"{LIB_PATH} has ABI version {lib.pkv_abi_version()}, "
                               f"this binding needs {ABI_VERSION}: rebuild")
        _lib = lib
        return lib


def _check(status: int):
    if status != PKV_OK:
        msg = load().pkv_last_error_message().decode(errors="replace")
        raise PkvError(status, msg)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(name: str, t: torch.Tensor, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise PkvError(1, f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise PkvError(1, f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise PkvError(1, f"{name} must be {dtype}, got {t.dtype}")


def _need_page_params(desc: CacheDesc, t: Optional[torch.Tensor], name: str):
    """E4M3: fp32 [S][NB][Hkv]; INT8: fp32 [S][NB][Hkv][2] (scale, zero)."""
    _need_cuda(name, t, torch.float32)
    want = (desc.num_slots, desc.num_blocks, desc.num_kv_heads)
    if desc.dtype == KV_INT8:
        want = want + (2,)
    if tuple(t.shape) != want:
        raise PkvError(1, f"{name} must have shape {list(want)}")


def cache_desc(k_cache: torch.Tensor) -> CacheDesc:
    """Descriptor of a [S][NB][Hkv][bs][D] cache tensor (bf16, or uint8 = E4M3)."""
    if k_cache.dim() != 5:
        raise PkvError(1, "cache must be 5-D [S][NB][Hkv][bs][D]")
    if k_cache.dtype == torch.bfloat16:
        dt = KV_BF16
    elif k_cache.dtype == torch.uint8:
        dt = KV_FP8_E4M3
    elif k_cache.dtype == torch.int8:
        dt = KV_INT8
    else:
        raise PkvError(1, f"cache dtype {k_cache.dtype} (bfloat16, uint8 E4M3 codes or int8)")
    S, NB, Hkv, bs, D = (int(x) for x in k_cache.shape)
    return CacheDesc(S, NB, bs, Hkv, D, dt)


def kv_append(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
              k_cache: torch.Tensor, v_cache: torch.Tensor,
              k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
              slot: int = 0, stream=None) -> None:
    """Write new tokens k, v [N][Hkv][D] (bf16) into cache slot ``slot`` at
    ``slot_mapping`` (int64 [N], -1 = skip)."""
    desc = cache_desc(k_cache)
    for n, t in (("k", k), ("v", v)):
        _need_cuda(n, t, torch.bfloat16)
    _need_cuda("slot_mapping", slot_mapping, torch.int64)
    _need_cuda("k_cache", k_cache)
    _need_cuda("v_cache", v_cache, k_cache.dtype)
    N = int(slot_mapping.shape[0])
    if k.shape != (N, desc.num_kv_heads, desc.head_dim) or v.shape != k.shape:
        raise PkvError(1, f"k/v must be [{N}][{desc.num_kv_heads}][{desc.head_dim}]")
    if desc.dtype != KV_BF16:
        _need_page_params(desc, k_scale, "k_scale")
        _need_page_params(desc, v_scale, "v_scale")
    _check(load().pkv_kv_append(ctypes.byref(desc), int(slot), _ptr(k), _ptr(v), _ptr(slot_mapping),
                                N, _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                _stream_handle(stream)))


def decode_opts(partition_blocks: int = 0, math: int = MATH_AUTO, warps: int = 0,
                stages: int = 0, event_start=None, event_end=None) -> DecodeOpts:
    """Options of :func:`paged_decode`.  ``event_start`` / ``event_end``:
    optional torch.cuda.Event objects recorded around the decode kernel."""
    def handle(ev):
        return None if ev is None else ctypes.c_void_p(ev.cuda_event)
    return DecodeOpts(int(partition_blocks), int(math), int(warps), int(stages),
                      handle(event_start), handle(event_end))


def decode_workspace_bytes(k_cache: torch.Tensor, batch: int, num_q_heads: int,
                           max_blocks_per_seq: int, opts: Optional[DecodeOpts] = None,
                           query_tokens: int = 1) -> int:
    desc = cache_desc(k_cache)
    n = load().pkv_decode_multi_workspace_bytes(ctypes.byref(desc), int(batch), int(query_tokens),
                                                int(num_q_heads), int(max_blocks_per_seq),
                                                ctypes.byref(opts) if opts is not None else None)
    if n == 0:
        raise PkvError(1, "bad arguments for the decode workspace")
    return int(n)


def decode_plan(k_cache: torch.Tensor, batch: int, num_q_heads: int, max_blocks_per_seq: int,
                opts: Optional[DecodeOpts] = None, query_tokens: int = 1) -> dict:
    """The resolved launch plan of a decode call (host only, nothing launched)."""
    desc = cache_desc(k_cache)
    plan = DecodePlan()
    _check(load().pkv_decode_multi_describe(ctypes.byref(desc), int(batch), int(query_tokens),
                                            int(num_q_heads), int(max_blocks_per_seq),
                                            ctypes.byref(opts) if opts is not None else None,
                                            ctypes.byref(plan)))
    return {f: getattr(plan, f) for f, _ in DecodePlan._fields_}


def new_decode_workspace(k_cache: torch.Tensor, batch: int, num_q_heads: int,
                         max_blocks_per_seq: int, opts: Optional[DecodeOpts] = None,
                         query_tokens: int = 1) -> torch.Tensor:
    """Zero-filled device workspace for :func:`paged_decode` (or, with
    ``query_tokens`` T, :func:`paged_decode_multi`)."""
    n = decode_workspace_bytes(k_cache, batch, num_q_heads, max_blocks_per_seq, opts, query_tokens)
    return torch.zeros(n, dtype=torch.uint8, device=k_cache.device)


def _marshal_decode(q, k_cache, v_cache, block_tables, context_lens, kv_group_ptr, layer, scale, out,
                    workspace, k_scale, v_scale, opts, k_new=None, v_new=None, slot_mapping=None,
                    want_dim=None):
    """Check one decode call's arguments and turn them into the C call's
    argument list (without the trailing stream).  Returns (function, args,
    out, workspace)."""
    desc = cache_desc(k_cache)
    _need_cuda("q", q, torch.bfloat16)
    _need_cuda("k_cache", k_cache)
    _need_cuda("v_cache", v_cache, k_cache.dtype)
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    if want_dim is not None and q.dim() != want_dim:
        raise PkvError(1, "q must be [B][Hq][D]" if want_dim == 3 else "q must be [B][T][Hq][D]")
    if q.dim() == 3:
        B, Hq, D = (int(x) for x in q.shape)
        T = 1
    elif q.dim() == 4:
        B, T, Hq, D = (int(x) for x in q.shape)
    else:
        raise PkvError(1, "q must be [B][Hq][D] or [B][T][Hq][D]")
    if D != desc.head_dim or block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise PkvError(1, "q / block_tables shapes do not match the cache")
    append = k_new is not None or v_new is not None or slot_mapping is not None
    if append:
        _need_cuda("k_new", k_new, torch.bfloat16)
        _need_cuda("v_new", v_new, torch.bfloat16)
        _need_cuda("slot_mapping", slot_mapping, torch.int64)
        N = int(slot_mapping.numel())
        if k_new.shape != (N, desc.num_kv_heads, desc.head_dim) or v_new.shape != k_new.shape:
            raise PkvError(1, "k_new / v_new must be [N][Hkv][D] with N = len(slot_mapping)")
    MB = int(block_tables.shape[1])
    if out is None:
        out = torch.empty_like(q)
    _need_cuda("out", out, torch.bfloat16)
    if out.shape != q.shape:
        raise PkvError(1, "out must be shaped like q")
    if desc.dtype != KV_BF16:
        _need_page_params(desc, k_scale, "k_scale")
        _need_page_params(desc, v_scale, "v_scale")
    if workspace is None:
        workspace = new_decode_workspace(k_cache, B, Hq, MB, opts, T)
    gp = (ctypes.c_int32 * len(kv_group_ptr))(*[int(x) for x in kv_group_ptr])
    if scale is None:
        scale = D ** -0.5
    popts = ctypes.byref(opts) if opts is not None else None
    tail = (_ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(block_tables), MB,
            _ptr(context_lens), gp, len(kv_group_ptr), int(layer), float(scale), _ptr(out),
            _ptr(workspace), int(workspace.numel()), popts)
    lib = load()
    if append:
        return (lib.pkv_append_and_decode,
                (ctypes.byref(desc), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), N, _ptr(q), B, T, Hq)
                + tail, out, workspace)
    if q.dim() == 4:
        return lib.pkv_paged_decode_multi, (ctypes.byref(desc), _ptr(q), B, T, Hq) + tail, out, workspace
    return lib.pkv_paged_decode, (ctypes.byref(desc), _ptr(q), B, Hq) + tail, out, workspace


def paged_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 block_tables: torch.Tensor, context_lens: torch.Tensor,
                 kv_group_ptr: Sequence[int] = (0,), layer: int = 0,
                 scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None,
                 k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
                 opts: Optional[DecodeOpts] = None, stream=None) -> torch.Tensor:
    """One decode step of one layer: returns out [B][Hq][D] (bf16)."""
    fn, args, out, _ = _marshal_decode(q, k_cache, v_cache, block_tables, context_lens, kv_group_ptr, layer,
                                       scale, out, workspace, k_scale, v_scale, opts, want_dim=3)
    _check(fn(*args, _stream_handle(stream)))
    return out


def paged_decode_multi(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                       block_tables: torch.Tensor, context_lens: torch.Tensor,
                       kv_group_ptr: Sequence[int] = (0,), layer: int = 0,
                       scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None,
                       k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
                       opts: Optional[DecodeOpts] = None, stream=None) -> torch.Tensor:
    """T new query tokens per sequence, q [B][T][Hq][D] (bf16), already
    appended as the last T cached tokens; token t attends causally to the
    first context_lens[b] - T + t + 1 tokens.  Returns out [B][T][Hq][D]."""
    fn, args, out, _ = _marshal_decode(q, k_cache, v_cache, block_tables, context_lens, kv_group_ptr, layer,
                                       scale, out, workspace, k_scale, v_scale, opts, want_dim=4)
    _check(fn(*args, _stream_handle(stream)))
    return out


def append_and_decode(k_new: torch.Tensor, v_new: torch.Tensor, slot_mapping: torch.Tensor,
                      q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_tables: torch.Tensor, context_lens: torch.Tensor,
                      kv_group_ptr: Sequence[int] = (0,), layer: int = 0,
                      scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None,
                      k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
                      opts: Optional[DecodeOpts] = None, stream=None) -> torch.Tensor:
    """One step in one call: :func:`kv_append` of k_new / v_new [N][Hkv][D]
    at ``slot_mapping`` into cache slot ``kv_group_ptr[layer]``, then
    :func:`paged_decode` (q [B][Hq][D]) or :func:`paged_decode_multi`
    (q [B][T][Hq][D]).  Returns out, shaped like q."""
    if k_new is None or v_new is None or slot_mapping is None:
        raise PkvError(1, "k_new, v_new and slot_mapping are required")
    fn, args, out, _ = _marshal_decode(q, k_cache, v_cache, block_tables, context_lens, kv_group_ptr, layer,
                                       scale, out, workspace, k_scale, v_scale, opts, k_new, v_new,
                                       slot_mapping)
    _check(fn(*args, _stream_handle(stream)))
    return out


class PreparedDecode:
    """A decode call (:func:`paged_decode`, :func:`paged_decode_multi`, or
    :func:`append_and_decode` when ``k_new`` / ``v_new`` / ``slot_mapping``
    are given) whose arguments were checked and marshalled once.  Each call
    of the object enqueues the same launch again, reading whatever the bound
    tensors hold at that time: the pattern of a serving loop whose step
    buffers stay in place (as under CUDA graph capture) and whose host cost
    per step must stay small.  The object keeps every bound tensor alive.
    ``stream``: the stream bound at preparation (default: the current stream
    at each call); a call may override it."""

    def __init__(self, q, k_cache, v_cache, block_tables, context_lens, kv_group_ptr=(0,), layer=0,
                 scale=None, out=None, workspace=None, k_scale=None, v_scale=None, opts=None,
                 k_new=None, v_new=None, slot_mapping=None, stream=None):
        fn, args, out, workspace = _marshal_decode(q, k_cache, v_cache, block_tables, context_lens,
                                                   kv_group_ptr, layer, scale, out, workspace, k_scale,
                                                   v_scale, opts, k_new, v_new, slot_mapping)
        self._fn, self._args = fn, args
        self._keep = (q, k_cache, v_cache, block_tables, context_lens, k_scale, v_scale, opts, k_new,
                      v_new, slot_mapping)
        self.out, self.workspace = out, workspace
        self._stream = None if stream is None else _stream_handle(stream)

    def __call__(self, stream=None) -> torch.Tensor:
        h = _stream_handle(stream) if (stream is not None or self._stream is None) else self._stream
        st = self._fn(*self._args, h)
        if st != PKV_OK:
            _check(st)
        return self.out


def copy_blocks(src_k: torch.Tensor, src_v: torch.Tensor, dst_k: torch.Tensor,
                dst_v: torch.Tensor, block_pairs: torch.Tensor,
                src_k_scale: Optional[torch.Tensor] = None, src_v_scale: Optional[torch.Tensor] = None,
                dst_k_scale: Optional[torch.Tensor] = None, dst_v_scale: Optional[torch.Tensor] = None,
                stream=None) -> None:
    """Copy blocks ``block_pairs[i] = (src, dst)`` (device int32 [n][2]) from
    one pool ``[NB][Hkv][bs][D]`` to another.  Pools may live in device
    memory or in pinned host memory (``tensor.pin_memory()``)."""
    for n, t in (("src_k", src_k), ("src_v", src_v), ("dst_k", dst_k), ("dst_v", dst_v)):
        if t.dim() != 4 or not t.is_contiguous():
            raise PkvError(1, f"{n} must be a contiguous [NB][Hkv][bs][D] tensor")
        if not (t.is_cuda or t.is_pinned()):
            raise PkvError(1, f"{n} must be a CUDA tensor or pinned host memory")
    if src_k.shape[1:] != dst_k.shape[1:] or src_k.dtype != dst_k.dtype:
        raise PkvError(1, "source and destination pages differ in shape or dtype")
    _need_cuda("block_pairs", block_pairs, torch.int32)
    desc = cache_desc(src_k.unsqueeze(0))
    n = int(block_pairs.shape[0])
    _check(load().pkv_copy_blocks(
        ctypes.byref(desc), _ptr(src_k), _ptr(src_v), _ptr(src_k_scale), _ptr(src_v_scale),
        int(src_k.shape[0]), _ptr(dst_k), _ptr(dst_v), _ptr(dst_k_scale), _ptr(dst_v_scale),
        int(dst_k.shape[0]), _ptr(block_pairs), n, _stream_handle(stream)))


STATIC_WORKSPACE_MAX_BYTES = 16 << 20


def paged_decode_static_workspace(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                  block_tables: torch.Tensor, context_lens: torch.Tensor,
                                  kv_group_ptr: Sequence[int] = (0,), layer: int = 0,
                                  scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                                  k_scale: Optional[torch.Tensor] = None,
                                  v_scale: Optional[torch.Tensor] = None,
                                  opts: Optional[DecodeOpts] = None, stream=None) -> torch.Tensor:
    """:func:`paged_decode` for callers that cannot allocate a workspace: the
    library's built-in static device array serves as scratch (at most
    STATIC_WORKSPACE_MAX_BYTES; calls that overlap on the GPU race on it).
    ``out`` must be passed in by a caller that cannot allocate."""
    desc = cache_desc(k_cache)
    _need_cuda("q", q, torch.bfloat16)
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    B, Hq, D = (int(x) for x in q.shape)
    if out is None:
        out = torch.empty_like(q)
    _need_cuda("out", out, torch.bfloat16)
    gp = (ctypes.c_int32 * len(kv_group_ptr))(*[int(x) for x in kv_group_ptr])
    if scale is None:
        scale = D ** -0.5
    _check(load().pkv_paged_decode_static_workspace(
        ctypes.byref(desc), _ptr(q), B, Hq, _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
        _ptr(v_scale), _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens), gp,
        len(kv_group_ptr), int(layer), float(scale), _ptr(out),
        ctypes.byref(opts) if opts is not None else None, _stream_handle(stream)))
    return out


def read_probe(data: torch.Tensor, sum_out: torch.Tensor, stream=None) -> torch.Tensor:
    """Read-only HBM probe (a measurement aid, not part of the decode): one
    launch streams the contiguous CUDA tensor ``data`` once and adds the
    unsigned sum of its 32-bit words, modulo 2^64, to ``sum_out`` (a CUDA
    int64 tensor of one element, holding the bits of a uint64)."""
    if not isinstance(data, torch.Tensor) or not data.is_cuda or not data.is_contiguous():
        raise PkvError(1, "data must be a contiguous CUDA tensor")
    _need_cuda("sum_out", sum_out, torch.int64)
    if sum_out.numel() != 1:
        raise PkvError(1, "sum_out must hold one element")
    _check(load().pkv_read_probe(_ptr(data), int(data.numel() * data.element_size()), _ptr(sum_out),
                                 _stream_handle(stream)))
    return sum_out


def read_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word."""
    flags = ctypes.c_uint32(0)
    st = load().pkv_read_device_error(ctypes.byref(flags), _stream_handle(stream))
    if st not in (PKV_OK, 5):
        _check(st)
    return int(flags.value)


def build(force: bool = False) -> str:
    from . import _build
    return _build.build(force=force)


# ---------------------------------------------------------------------------
# prefix cache (host only; include/pkv_prefix.h)
# ---------------------------------------------------------------------------
def _i32_array(values) -> "ctypes.Array":
    vals = [int(v) for v in values]
    return (ctypes.c_int32 * max(1, len(vals)))(*vals)


def prefix_block_hashes(tokens: Sequence[int], block_size: int) -> list:
    """Cumulative FNV-1a-64 hash of every full block of a token sequence."""
    n = len(tokens)
    nb = n // int(block_size) if block_size > 0 else 0
    out = (ctypes.c_uint64 * max(1, nb))()
    _check(load().pkv_prefix_block_hashes(int(block_size), _i32_array(tokens), n, out))
    return [int(out[j]) for j in range(nb)]


class PrefixCache:
    """Host index from block content to physical block, per layer group:
    ``match`` walks a request's full blocks and returns the physical blocks of
    its cached prefix; ``insert`` registers a sequence's full blocks; ``erase``
    forgets freed blocks."""

    def __init__(self, block_size: int, num_groups: int = 1):
        self._lib = load()
        h = ctypes.c_void_p()
        _check(self._lib.pkv_prefix_cache_create(int(block_size), int(num_groups), ctypes.byref(h)))
        self._h = h
        self.block_size = int(block_size)

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.pkv_prefix_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def match(self, tokens: Sequence[int], group: int = 0, max_blocks: Optional[int] = None) -> list:
        nb = len(tokens) // self.block_size
        cap = nb if max_blocks is None else min(nb, int(max_blocks))
        ids = (ctypes.c_int32 * max(1, cap))()
        n = ctypes.c_int32(0)
        _check(self._lib.pkv_prefix_cache_match(self._h, int(group), _i32_array(tokens), len(tokens), ids,
                                                 cap, ctypes.byref(n)))
        return [int(ids[j]) for j in range(n.value)]

    def insert(self, tokens: Sequence[int], block_ids: Sequence[int], group: int = 0) -> int:
        n = ctypes.c_int32(0)
        _check(self._lib.pkv_prefix_cache_insert(self._h, int(group), _i32_array(tokens), len(tokens),
                                                  _i32_array(block_ids), len(block_ids), ctypes.byref(n)))
        return n.value

    def erase(self, block_ids: Sequence[int], group: int = 0) -> int:
        n = ctypes.c_int32(0)
        _check(self._lib.pkv_prefix_cache_erase(self._h, int(group), _i32_array(block_ids), len(block_ids),
                                                 ctypes.byref(n)))
        return n.value

    def stats(self, group: int = 0):
        """(entries, lookups, hits) of one group."""
        e, l, h = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
        _check(self._lib.pkv_prefix_cache_stats(self._h, int(group), ctypes.byref(e), ctypes.byref(l),
                                                 ctypes.byref(h)))
        return e.value, l.value, h.value
