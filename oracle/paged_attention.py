"""Paged decode attention, restated in float64.

Definition followed (cs2680 Lecture 10, §10.3 "PagedAttention: the KV cache as
virtual memory"; "KV cache systems", block-table indirection paragraph):
token t of sequence s lives in physical block block_table[s][t // b] at row
t mod b, and decode attention of the single new query over the first
context_len[s] tokens is

    x_t = scale * <q[s, h], K[s, g(h), t]>
    o[s, h] = sum_t exp(x_t - max x) V[s, g(h), t] / sum_t exp(x_t - max x)

Paging changes neither the FLOPs nor the bytes, only where the kernel reads
them (§10.3, step three), so this is ordinary attention over the gathered
rows. Readings where the pages are silent:
  - grouped-query mapping: query head h uses KV head h // (Hq / Hkv);
  - context_len == 0 gives an all-zero output;
  - cache layout [num_blocks, Hkv, b, D]; entries past ceil(ctx / b) in a
    block-table row are never read.
"""
from __future__ import annotations

import numpy as np


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    u32 = bits.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def gather_tokens(cache: np.ndarray, table_row: np.ndarray, ctx: int, kv_head: int) -> np.ndarray:
    """Rows [ctx, D] (float64) of one sequence and KV head, read through its table."""
    b = cache.shape[2]
    t = np.arange(ctx)
    phys = table_row[t // b]
    return widen_bf16(cache[phys, kv_head, t % b, :])


def attend_one(q_vec: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float) -> np.ndarray:
    """softmax(scale * keys @ q) @ values for one query vector (float64)."""
    x = scale * np.einsum("td,d->t", keys, q_vec)
    w = np.exp(x - x.max())
    return np.einsum("t,td->d", w, values) / w.sum()


def paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale, seqs=None):
    """Decode attention for every (sequence, query head); returns float64 [B, Hq, D].

    q: uint16 [B, Hq, D]; k_cache, v_cache: uint16 [NB, Hkv, b, D];
    block_tables: int [B, W]; context_lens: int [B]. `seqs` restricts the
    computation to the listed sequences (other rows stay zero).
    """
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D), dtype=np.float64)
    qf = widen_bf16(q)
    for s in range(B) if seqs is None else seqs:
        n = int(context_lens[s])
        if n <= 0:
            continue
        for g in range(Hkv):
            keys = gather_tokens(k_cache, block_tables[s], n, g)
            values = gather_tokens(v_cache, block_tables[s], n, g)
            for h in range(g * G, (g + 1) * G):
                out[s, h] = attend_one(qf[s, h], keys, values, scale)
    return out


def partitioned_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale, partition_tokens):
    """The same attention computed in context partitions of `partition_tokens`
    tokens, each reduced to (m, l, a) = (max logit, sum exp(x - m),
    sum exp(x - m) v), then combined with a log-sum-exp rescale:
        M = max_p m_p,  o = sum_p e^(m_p - M) a_p / sum_p e^(m_p - M) l_p.
    Algebraically identical to paged_decode_attention."""
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    G = Hq // Hkv
    P = int(partition_tokens)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    qf = widen_bf16(q)
    for s in range(B):
        n = int(context_lens[s])
        if n <= 0:
            continue
        for g in range(Hkv):
            keys = gather_tokens(k_cache, block_tables[s], n, g)
            values = gather_tokens(v_cache, block_tables[s], n, g)
            for h in range(g * G, (g + 1) * G):
                parts = []
                for lo in range(0, n, P):
                    x = scale * np.einsum("td,d->t", keys[lo : lo + P], qf[s, h])
                    m = x.max()
                    e = np.exp(x - m)
                    parts.append((m, e.sum(), np.einsum("t,td->d", e, values[lo : lo + P])))
                M = max(p[0] for p in parts)
                num = sum(np.exp(m - M) * a for m, _, a in parts)
                den = sum(np.exp(m - M) * l for m, l, _ in parts)
                out[s, h] = num / den
    return out
