/*
 * pkv -- paged KV-cache decode attention for NVIDIA GB300 (sm_103a).
 *
 * C ABI.  Every pointer argument is a plain address; "device" pointers are
 * CUDA device (or managed) memory owned by the caller, "host" pointers are
 * ordinary host memory owned by the caller.  The library keeps no reference
 * to any argument after a call returns.  All GPU work is enqueued on the
 * caller's stream (`stream` is a cudaStream_t; NULL = the legacy default
 * stream) and runs asynchronously; a PKV_OK return means "validated and
 * launched", not "finished".
 *
 * Citations name the web page and section the operation comes from:
 *   [BW] "KV Cache Engineering: PagedAttention, Continuous Batching,
 *        Attention Variants, and the Bandwidth Wall"
 *   [PC] "KV-Cache Engineering: Paged Attention, Prefix Cache,
 *        Disaggregation (2026)"
 *
 * Data layout (the pages draw physical blocks as opaque boxes; this layout
 * is the library's choice):
 *   k_cache, v_cache  [S][NB][Hkv][bs][D]   S cache slots (layer groups),
 *                     NB physical blocks, Hkv KV heads, bs tokens per block,
 *                     D head_dim.  Element type bf16, FP8 E4M3 or INT8
 *                     (1 byte).
 *                     One (slot, block, KV head) page is a contiguous
 *                     bs*D run.
 *   k_scale, v_scale  E4M3 caches: fp32 [S][NB][Hkv], one scale per page;
 *                     stored value = e4m3(x / scale).
 *                     INT8 caches: fp32 [S][NB][Hkv][2], (scale, zero point)
 *                     per page, the zero point an integer in [-128, 127];
 *                     stored value q = clamp(rne(x / scale) + zero, lo, 127)
 *                     with lo = -127 when zero == 0 (symmetric) and -128
 *                     otherwise; value read back = (q - zero) * scale.
 *                     Alignment: 4 bytes (E4M3) or 8 bytes (INT8), else
 *                     PKV_ERR_ALIGNMENT.
 *                     Source: [BW] "INT8 KV cache" (symmetric or asymmetric
 *                     quantisation with a scale and zero point).
 *   q, out            bf16 [B][Hq][D]       one query token per sequence.
 *   block_tables      int32 [B][MB]         logical block j of sequence b is
 *                     physical block block_tables[b*MB + j].
 *   context_lens      int32 [B]             tokens sequence b attends to,
 *                     including the token appended this step; 0 = inactive.
 * Query head h belongs to KV head h / G with G = Hq / Hkv (contiguous GQA
 * groups; G = 1 is MHA, Hkv = 1 is MQA).
 *
 * Errors.  Argument problems the host can see (null or misaligned pointers,
 * unsupported shapes, a shared-with pointer outside the slots, a workspace
 * that is too small) return a status before anything is launched.
 * Problems only the data shows (a block id outside [0, NB), a slot outside
 * [-1, NB*bs), a context length outside [0, MB*bs]) are skipped on the
 * device: the offending page, token or sequence contributes nothing, and a
 * sticky device error word records the kind of fault; read it with
 * pkv_read_device_error().  Kernels never trap.  With the environment
 * variable PKV_VALIDATE=1 the host also copies the tables back and checks
 * them before launching (slow; synchronises the stream).
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_ABI_VERSION 2

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,   /* null pointer, bad size, bad index argument */
  PKV_ERR_UNSUPPORTED = 2,   /* shape or dtype this build has no kernel for */
  PKV_ERR_ALIGNMENT = 3,     /* a tensor is not aligned as its call requires */
  PKV_ERR_CUDA = 4,          /* a CUDA runtime/driver call or launch failed */
  PKV_ERR_DEVICE_INDEX = 5,  /* the device error word was non-zero */
  PKV_ERR_WORKSPACE = 6      /* workspace missing or smaller than required */
} pkv_status;

typedef enum { PKV_KV_BF16 = 0, PKV_KV_FP8_E4M3 = 1, PKV_KV_INT8 = 2 } pkv_kv_dtype;

/* Bits of the device error word. */
#define PKV_DEVERR_BLOCK_ID 0x1u     /* block table entry outside [0, NB) */
#define PKV_DEVERR_SLOT 0x2u         /* slot_mapping entry outside [-1, NB*bs) */
#define PKV_DEVERR_CONTEXT_LEN 0x4u  /* context length outside [0, MB*bs] */
#define PKV_DEVERR_TIMEOUT 0x8u      /* a bounded wait on a copy gave up */

/* Shape of one paged cache (both K and V).  Supported: block_size 16 or 32;
 * head_dim 64 or 128 for bf16, 128 for E4M3 and INT8. */
typedef struct {
  int32_t num_slots;    /* S: independent caches (layer groups) */
  int32_t num_blocks;   /* NB: physical blocks per slot */
  int32_t block_size;   /* bs: tokens per block */
  int32_t num_kv_heads; /* Hkv */
  int32_t head_dim;     /* D */
  int32_t dtype;        /* pkv_kv_dtype */
} pkv_cache_desc;

/* How the decode computes its dot products. */
typedef enum {
  PKV_MATH_AUTO = 0, /* the library picks: TC for multi-token calls with more
                        than 16 query rows per KV head and head_dim 128, else MMA */
  PKV_MATH_FFMA = 1, /* fp32 CUDA-core FMAs; G must be 1, 2, 4 or 8; T = 1 */
  PKV_MATH_MMA = 2,  /* mma.sync tiles of up to 16 rows (bf16, or f16 for one-byte
                        caches); G <= 16 */
  PKV_MATH_TC = 3    /* tcgen05 tiles of 128 (query token, head) rows with TMEM
                        accumulators; multi-token calls (T > 1), head_dim 128,
                        G <= 128; bf16 pages as they are; E4M3 K pages as
                        they are (E4M3 products against a two-part E4M3
                        query), INT8 K and all one-byte V pages as f16 code
                        values, with the page scales applied to the scores
                        and to P; with more than one tile per KV head
                        (bf16), pairs of tiles share each page read */
} pkv_decode_math;

/* Tuning knobs of pkv_paged_decode; a NULL pointer or zero fields = auto. */
typedef struct {
  int32_t partition_blocks; /* blocks per split-K partition, 1..64, or 1..256 for
                               PKV_MATH_TC (0 = auto; auto may take 128 or 256 for
                               PKV_MATH_TC); with automatic partitions the tile-pair
                               tcgen05 kernel may give the last sequences
                               partitions of half this length, so that the
                               last round of its units is not left under half
                               full */
  int32_t math;             /* pkv_decode_math */
  int32_t warps_per_cta;    /* 1..8 (0 = auto) */
  int32_t stages;           /* pages in each warp's copy ring, 2..8 (0 = auto) */
  /* Optional cudaEvent_t handles (NULL = none) that the library records on
   * the stream immediately before and after the decode kernel itself (not
   * the planner), for timing that one kernel.  Recording the start event
   * between the two kernels keeps them from overlapping. */
  void* event_decode_start;
  void* event_decode_end;
} pkv_decode_opts;

/*
 * Write new tokens' K and V into their physical slots.
 * Source: [BW] "What the KV Cache Stores and Why" (each step computes K and
 * V for the new token only and stores them) and "Continuous Batching" (a
 * growing sequence takes blocks from the free pool).
 *
 *   cache        shape of k_cache / v_cache (host).
 *   slot         cache slot (layer group) to write, in [0, S).
 *   k, v         device bf16 [N][Hkv][D]: the new tokens.
 *   slot_mapping device int64 [N]: physical block * bs + offset; -1 skips the
 *                token (padding).  Other out-of-range values set
 *                PKV_DEVERR_SLOT and skip the token.  Two tokens with the
 *                same slot in one call: unspecified which one lands.
 *   k_cache, v_cache  device, written in place.
 *   k_scale, v_scale  device, E4M3 and INT8 caches only (may be NULL for
 *                bf16), layouts as above: E4M3 byte =
 *                e4m3_rn_satfinite(float(x) / scale); INT8 byte = clamp(rne(
 *                float(x) / scale) + zero, lo, 127).  The division is IEEE
 *                binary32.  bf16 caches receive the bits as is.
 * Returns PKV_OK after launching one kernel (none when N == 0).
 */
pkv_status pkv_kv_append(const pkv_cache_desc* cache, int32_t slot,
                         const void* k, const void* v, const int64_t* slot_mapping,
                         int32_t num_tokens, void* k_cache, void* v_cache,
                         const float* k_scale, const float* v_scale, void* stream);

/*
 * Bytes of device workspace pkv_paged_decode needs for these sizes (0 on a
 * bad argument).  The workspace holds the split-K partials, the per-call
 * plan (partition prefix sums, validated context lengths) and a work-queue
 * counter.  It needs no initialisation: each call's planner kernel writes
 * every field before the decode reads it.  Calls that may run at the same
 * time (different streams) need separate workspaces.
 */
size_t pkv_decode_workspace_bytes(const pkv_cache_desc* cache, int32_t batch,
                                  int32_t num_q_heads, int32_t max_blocks_per_seq,
                                  const pkv_decode_opts* opts);

/* The launch plan pkv_paged_decode would use for these sizes and options. */
typedef struct {
  int32_t partition_blocks;  /* blocks per split-K partition */
  int32_t max_partitions;    /* partitions of a max_blocks_per_seq-block sequence
                                (at half-length partitions where those apply) */
  int32_t math;              /* resolved pkv_decode_math */
  int32_t warps_per_cta;
  int32_t stages;
  int32_t kernels_per_call;  /* planner + decode (+ merge above 4 partitions) */
  size_t workspace_bytes;
  size_t smem_bytes_per_cta;
  int32_t query_tokens_per_tile; /* multi-token queries: tokens per row tile (1 for T = 1) */
  int32_t row_tiles;             /* row tiles per (sequence, KV head): each reads the pages */
} pkv_decode_plan;

/*
 * Resolve the options of a decode call without launching anything (host
 * only).  Same argument checks as pkv_paged_decode's shape checks; *plan is
 * written on PKV_OK.
 */
pkv_status pkv_decode_describe(const pkv_cache_desc* cache, int32_t batch, int32_t num_q_heads,
                               int32_t max_blocks_per_seq, const pkv_decode_opts* opts,
                               pkv_decode_plan* plan);

/*
 * Single-token decode attention over the paged cache, one query token per
 * sequence:
 *   out[b][h][:] = sum_t softmax_t(scale * q[b][h] . K_t) V_t,
 *   t = 0 .. context_lens[b]-1, K_t = k_cache[slot][block_tables[b][t/bs]]
 *   [h/G][t%bs] (V_t alike), slot = kv_group_ptr[layer].
 * Sources: [BW] "What the KV Cache Stores and Why" (attend the new Q over all
 * cached K,V), "PagedAttention" (block table maps logical to physical
 * blocks; only the last block is partly filled), "Attention Variants"
 * (grouped-query heads), "FP8 KV cache" (dequantise on read); [PC]
 * cross-layer KV sharing Q&A (each logical layer has a shared-with pointer
 * naming its group's cache).
 *
 *   q              device bf16 [B][Hq][D].
 *   k/v_cache      device [S][NB][Hkv][bs][D] as described by `cache`.
 *   k/v_scale      device, E4M3 / INT8 only (NULL for bf16), layouts as above.
 *   block_tables   device int32 [B][max_blocks_per_seq]; entries past a
 *                  sequence's last block are never read.
 *   context_lens   device int32 [B].
 *   kv_group_ptr   HOST int32 [num_layers]: the cache slot layer l reads
 *                  (the shared-with pointer); layers of one group name the
 *                  same slot.  `layer` selects the entry for this call.
 *   scale          softmax scale applied to the fp32 logits (e.g. 1/sqrt(D)).
 *   out            device bf16 [B][Hq][D]; must not overlap q.  Sequences with
 *                  context_lens 0 get zeros.
 *   workspace      device, pkv_decode_workspace_bytes() bytes, see there.
 * Accumulation is fp32; out is rounded to bf16 (round to nearest even).
 * The reduction order depends only on logical token positions and the
 * partition size, never on which physical blocks hold the tokens.
 * Launches a planner and the decode kernel.  Sequences split into at most 4
 * partitions are merged by the decode warp that finishes last; with more
 * partitions a third kernel merges the partials.  Both kernels (and pkv_kv_append's) use programmatic dependent
 * launch: each may be scheduled while the previous kernel on the stream
 * drains, and waits for it before reading memory (PKV_PDL=0 turns this off).
 */
pkv_status pkv_paged_decode(const pkv_cache_desc* cache,
                            const void* q, int32_t batch, int32_t num_q_heads,
                            const void* k_cache, const void* v_cache,
                            const float* k_scale, const float* v_scale,
                            const int32_t* block_tables, int32_t max_blocks_per_seq,
                            const int32_t* context_lens,
                            const int32_t* kv_group_ptr, int32_t num_layers, int32_t layer,
                            float scale, void* out,
                            void* workspace, size_t workspace_bytes,
                            const pkv_decode_opts* opts, void* stream);

/* Largest number of query tokens per sequence of pkv_paged_decode_multi. */
#define PKV_MAX_QUERY_TOKENS 512

/*
 * Decode with T >= 1 new query tokens per sequence (T = 1 is
 * pkv_paged_decode): the verification step of speculative decoding, where
 * the target model checks T proposed tokens in one pass over the shared
 * cache ([PC] "How does speculative decoding interact with KV-cache
 * compression?"), and small prefill chunks over a paged cache ([BW]
 * "Continuous Batching", chunked prefill).  The T new tokens' K and V must
 * already be in the cache as the last T of the context_lens[b] tokens;
 * query token t (0..T-1) sits at position n - T + t (n = context_lens[b])
 * and attends causally to positions 0 .. n - T + t:
 *   out[b][t][h][:] = sum_j softmax_j(scale * q[b][t][h] . K_j) V_j,
 *   j = 0 .. n - T + t.
 * Rows with no position to attend to (n - T + t < 0, including n = 0) get
 * zeros.
 *
 *   q, out         device bf16 [B][T][Hq][D] (must not overlap).
 *   workspace      pkv_decode_multi_workspace_bytes() bytes.
 *   everything else as in pkv_paged_decode.
 * The tensor-core back-ends only (PKV_MATH_FFMA with T > 1 gives
 * PKV_ERR_UNSUPPORTED).  The (query token, head) rows of one KV head form
 * row tiles of whole query tokens: at most 16 rows for PKV_MATH_MMA, each
 * tile a separate stream over the pages (G * T <= 16 reads the cache once);
 * 128 rows for PKV_MATH_TC, where a KV head with two or more tiles is served
 * by CTAs that each hold a pair of its tiles and read every page once for
 * both.
 */
pkv_status pkv_paged_decode_multi(const pkv_cache_desc* cache,
                                  const void* q, int32_t batch, int32_t num_query_tokens,
                                  int32_t num_q_heads,
                                  const void* k_cache, const void* v_cache,
                                  const float* k_scale, const float* v_scale,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* context_lens,
                                  const int32_t* kv_group_ptr, int32_t num_layers, int32_t layer,
                                  float scale, void* out,
                                  void* workspace, size_t workspace_bytes,
                                  const pkv_decode_opts* opts, void* stream);

/*
 * One decode step in one call: append the step's new tokens into cache slot
 * kv_group_ptr[layer] (exactly pkv_kv_append with that slot), then decode
 * (exactly pkv_paged_decode_multi; num_query_tokens = 1 is pkv_paged_decode).
 * The append runs on extra CTAs of the decode's planner launch, so the step
 * costs one launch less and the append and the planning overlap.
 * Sources: [BW] "What the KV Cache Stores and Why" (a step stores the new
 * token's K,V, then attends over the whole cache).
 *
 *   k_new, v_new, slot_mapping, num_new_tokens   as pkv_kv_append's k, v,
 *                  slot_mapping, num_tokens (0: no append).
 *   everything else as in pkv_paged_decode_multi; k_cache and v_cache are
 *                  written (the append) before they are read.
 * Same results, bit for bit, as the two separate calls.
 */
pkv_status pkv_append_and_decode(const pkv_cache_desc* cache,
                                 const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                 int32_t num_new_tokens,
                                 const void* q, int32_t batch, int32_t num_query_tokens,
                                 int32_t num_q_heads,
                                 void* k_cache, void* v_cache,
                                 const float* k_scale, const float* v_scale,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* context_lens,
                                 const int32_t* kv_group_ptr, int32_t num_layers, int32_t layer,
                                 float scale, void* out,
                                 void* workspace, size_t workspace_bytes,
                                 const pkv_decode_opts* opts, void* stream);

/* Workspace bytes and launch plan of pkv_paged_decode_multi (0 / an error
 * status for invalid arguments), as for the single-token calls. */
size_t pkv_decode_multi_workspace_bytes(const pkv_cache_desc* cache, int32_t batch,
                                        int32_t num_query_tokens, int32_t num_q_heads,
                                        int32_t max_blocks_per_seq, const pkv_decode_opts* opts);
pkv_status pkv_decode_multi_describe(const pkv_cache_desc* cache, int32_t batch,
                                     int32_t num_query_tokens, int32_t num_q_heads,
                                     int32_t max_blocks_per_seq, const pkv_decode_opts* opts,
                                     pkv_decode_plan* plan);

/* Size of the library's built-in decode workspace (see below). */
#define PKV_STATIC_WORKSPACE_MAX_BYTES ((size_t)16 << 20)

/*
 * pkv_paged_decode without a caller workspace.  The web pages have no
 * counterpart to this call; it exists for callers that cannot allocate
 * device memory at the point where they decode: code running where
 * cudaMalloc is off limits (an allocator-free runtime, a plugin handed
 * only its input and output buffers, a host that owns every allocation).
 *
 * The scratch the decode needs (split-K partials, the per-call plan, the
 * work-queue counter) lives instead in one static device array of
 * PKV_STATIC_WORKSPACE_MAX_BYTES bytes that every GPU which loads the
 * library holds until the process exits.  Arguments and results are those of
 * pkv_paged_decode; q, caches, tables and out are still the caller's.
 *   - A request whose workspace (pkv_decode_workspace_bytes) would exceed
 *     the array returns PKV_ERR_WORKSPACE and launches nothing; larger
 *     opts->partition_blocks means fewer split-K partials.
 *   - The first call on a device looks up that device's copy of the array
 *     (cudaGetSymbolAddress, with the device current); make that first call
 *     before any stream capture on the device.  The address is kept per
 *     device together with the CUDA context it belongs to; a call made under
 *     another context (after cudaDeviceReset, or once the primary context was
 *     released and made again) looks it up anew, so that call too should come
 *     before any stream capture.
 *   - The call allocates nothing (no cudaMalloc / cudaFree).  Every call on
 *     a device shares the one array and it keeps the previous call's
 *     contents; each call's planner kernel rewrites everything the decode
 *     reads, so nothing needs clearing by the caller.  Calls that can run at
 *     the same time on the GPU (e.g. on different streams) race on the array.
 */
pkv_status pkv_paged_decode_static_workspace(const pkv_cache_desc* cache,
                                             const void* q, int32_t batch, int32_t num_q_heads,
                                             const void* k_cache, const void* v_cache,
                                             const float* k_scale, const float* v_scale,
                                             const int32_t* block_tables,
                                             int32_t max_blocks_per_seq,
                                             const int32_t* context_lens,
                                             const int32_t* kv_group_ptr, int32_t num_layers,
                                             int32_t layer, float scale, void* out,
                                             const pkv_decode_opts* opts, void* stream);

/*
 * Copy whole physical blocks between two block pools of the same page shape
 * (`cache` gives bs, Hkv, D and dtype; num_slots and num_blocks are not
 * used).  For each pair i, block src_ids[i] of the source pool is copied to
 * block dst_ids[i] of the destination pool: every KV head's K and V page
 * and, for E4M3 and INT8 pools, its K and V page parameters.
 * Sources: [BW] "PagedAttention" (block sharing: a sequence that appends
 * into a shared block first needs its own copy) and "KV-Cache Engineering:
 * The Memory Wall of LLM Serving", "Lever 5: Offloading" and "When the cache
 * fills" (moving a sequence's blocks to host memory and back).
 *
 *   src_k, src_v     source pool, [src_num_blocks][Hkv][bs][D]: device memory,
 *                    or host memory the GPU can address (pinned memory; on
 *                    systems with a coherent CPU-GPU interconnect any host
 *                    memory).  Point them at the first block of a cache slot.
 *   dst_k, dst_v     destination pool, [dst_num_blocks][Hkv][bs][D], same rules.
 *   src/dst_k_scale, src/dst_v_scale  fp32 [num_blocks][Hkv] (E4M3) or
 *                    [num_blocks][Hkv][2] (INT8, (scale, zero)); NULL for bf16.
 *   block_pairs      device int32 [count][2]: (src id, dst id).  Ids outside
 *                    their pool set PKV_DEVERR_BLOCK_ID and the pair is
 *                    skipped.  Two pairs with the same destination, or a
 *                    destination that is also a source of the same call:
 *                    unspecified result (validate mode rejects the first).
 * Bytes move unchanged (bit-exact).  One kernel launch (none when count == 0).
 */
pkv_status pkv_copy_blocks(const pkv_cache_desc* cache,
                           const void* src_k, const void* src_v, const float* src_k_scale,
                           const float* src_v_scale, int32_t src_num_blocks,
                           void* dst_k, void* dst_v, float* dst_k_scale, float* dst_v_scale,
                           int32_t dst_num_blocks, const int32_t* block_pairs, int32_t count,
                           void* stream);

/*
 * Read-only HBM probe, a measurement aid beside the decode (not part of it):
 * one kernel launch on `stream` reads `bytes` bytes at `data` once, with
 * 16-byte streaming loads, and adds the sum of their 32-bit words (unsigned,
 * modulo 2^64) to *sum.  The decode reads its cache and writes almost
 * nothing, so its ceiling is the read-only rate; this probe measures that
 * rate on the same device ("KV Cache Engineering: PagedAttention, Continuous
 * Batching, Attention Variants, and the Bandwidth Wall", "Two Costs:
 * Capacity and Bandwidth").
 *   data   device memory, 16-byte aligned, caller-owned, only read.
 *   bytes  a multiple of 16 (0: nothing is launched).
 *   sum    device uint64, 8-byte aligned, caller-owned; added to, not set.
 * Errors: NULL pointers or a size that is not a multiple of 16 ->
 * PKV_ERR_INVALID_ARG; misaligned pointers -> PKV_ERR_ALIGNMENT; a failed
 * launch -> PKV_ERR_CUDA.
 */
pkv_status pkv_read_probe(const void* data, size_t bytes, uint64_t* sum, void* stream);

/*
 * Synchronise `stream`, copy the current device's sticky error word into
 * *flags (PKV_DEVERR_* bits) and clear it.  Returns PKV_ERR_DEVICE_INDEX if
 * it was non-zero, PKV_OK if it was zero.
 */
pkv_status pkv_read_device_error(uint32_t* flags, void* stream);

/* Static text for a status code. */
const char* pkv_status_string(pkv_status status);

/* Text of the last error on the calling thread (host validation or CUDA). */
const char* pkv_last_error_message(void);

/* PKV_ABI_VERSION of the built library. */
int32_t pkv_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
