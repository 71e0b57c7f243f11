"""Test-side helpers that build paged caches from dense logical sequences.

The direction here is the opposite of the oracle's: a dense per-sequence
K/V array is *scattered* into randomly chosen physical blocks, and the block
table records where each logical block went.  References computed on the
dense arrays (torch SDPA in float64) are therefore independent of the
oracle's gather.
"""
import numpy as np
import torch

from workloads import bf16_bits_to_f32, normal_bf16_bits


def paged_from_dense(k_seqs, v_seqs, bs, seed, spare=3, fill=0, slots=1, slot=0, MB=None):
    """k_seqs[b]: array [n_b][Hkv][D] (any dtype).  Returns (k_cache, v_cache,
    block_tables, context_lens, placement) with caches [slots][NB][Hkv][bs][D]
    and placement[b] = list of physical blocks."""
    B = len(k_seqs)
    Hkv, D = k_seqs[0].shape[1], k_seqs[0].shape[2]
    dtype = k_seqs[0].dtype
    nblk = [-(-len(k) // bs) for k in k_seqs]
    NB = sum(nblk) + spare
    rng = np.random.Generator(np.random.PCG64(seed))
    perm = rng.permutation(NB)
    mb = MB if MB is not None else max(1, max(nblk))
    tables = np.full((B, mb), -1, dtype=np.int32)
    kc = np.full((slots, NB, Hkv, bs, D), fill, dtype=dtype)
    vc = np.full((slots, NB, Hkv, bs, D), fill, dtype=dtype)
    placement = []
    pos = 0
    for b in range(B):
        pl = []
        for j in range(nblk[b]):
            p = int(perm[pos])
            pos += 1
            tables[b, j] = p
            rows_k = k_seqs[b][j * bs:(j + 1) * bs]
            rows_v = v_seqs[b][j * bs:(j + 1) * bs]
            kc[slot, p, :, :len(rows_k), :] = np.transpose(rows_k, (1, 0, 2))
            vc[slot, p, :, :len(rows_v), :] = np.transpose(rows_v, (1, 0, 2))
            pl.append(p)
        placement.append(pl)
    ctx = np.array([len(k) for k in k_seqs], dtype=np.int32)
    return kc, vc, tables, ctx, placement


def dense_bf16_seqs(seed, lens, Hkv, D):
    ks = [normal_bf16_bits(seed * 31 + 2 + 1000 * i, (n, Hkv, D)) for i, n in enumerate(lens)]
    vs = [normal_bf16_bits(seed * 31 + 3 + 1000 * i, (n, Hkv, D)) for i, n in enumerate(lens)]
    return ks, vs


def sdpa_reference(q_bits, k_vals, v_vals, scale):
    """float64 torch SDPA per sequence on dense values.

    q_bits: bf16 bits [B][Hq][D]; k_vals[b], v_vals[b]: float64 [n][Hkv][D].
    GQA via enable_gqa (query head h reads KV head h // (Hq/Hkv))."""
    q = bf16_bits_to_f32(q_bits).astype(np.float64)
    B, Hq, D = q.shape
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        n = k_vals[b].shape[0]
        if n == 0:
            continue
        Hkv = k_vals[b].shape[1]
        qt = torch.from_numpy(q[b]).reshape(1, Hq, 1, D)
        kt = torch.from_numpy(np.ascontiguousarray(np.transpose(k_vals[b], (1, 0, 2)))).reshape(1, Hkv, n, D)
        vt = torch.from_numpy(np.ascontiguousarray(np.transpose(v_vals[b], (1, 0, 2)))).reshape(1, Hkv, n, D)
        o = torch.nn.functional.scaled_dot_product_attention(
            qt, kt, vt, scale=float(np.float32(scale)), enable_gqa=(Hkv != Hq))
        out[b] = o.reshape(Hq, D).numpy()
    return out


def sdpa_causal_tail_reference(q_bits, k_vals, v_vals, scale):
    """float64 torch SDPA for T new query tokens per sequence.

    q_bits: bf16 bits [B][T][Hq][D]; k_vals[b], v_vals[b]: float64 [n][Hkv][D]
    whose last T rows are the new tokens' keys and values.  The query tokens
    are placed at the last T positions of a square causal problem over all n
    positions (the earlier positions get zero queries, and their rows are
    dropped), so token t sees positions 0 .. n - T + t.  Rows whose position
    would be negative (n < T) are zero."""
    q = bf16_bits_to_f32(q_bits).astype(np.float64)
    B, T, Hq, D = q.shape
    out = np.zeros((B, T, Hq, D), dtype=np.float64)
    for b in range(B):
        n = k_vals[b].shape[0]
        if n == 0:
            continue
        Hkv = k_vals[b].shape[1]
        take = min(T, n)  # the last `take` query tokens have a position
        qf = np.zeros((n, Hq, D))
        qf[n - take:] = q[b, T - take:]
        qt = torch.from_numpy(np.ascontiguousarray(np.transpose(qf, (1, 0, 2)))).reshape(1, Hq, n, D)
        kt = torch.from_numpy(np.ascontiguousarray(np.transpose(k_vals[b], (1, 0, 2)))).reshape(1, Hkv, n, D)
        vt = torch.from_numpy(np.ascontiguousarray(np.transpose(v_vals[b], (1, 0, 2)))).reshape(1, Hkv, n, D)
        o = torch.nn.functional.scaled_dot_product_attention(
            qt, kt, vt, scale=float(np.float32(scale)), is_causal=True, enable_gqa=(Hkv != Hq))
        o = o.reshape(Hq, n, D).numpy()
        out[b, T - take:] = np.transpose(o[:, n - take:], (1, 0, 2))
    return out


def torch_e4m3_to_f64(codes):
    """Library decode of E4M3 codes (torch float8_e4m3fn) to float64."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_f32_to_e4m3(x):
    """Library E4M3 rounding (torch float8_e4m3fn, round-to-nearest-even)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
