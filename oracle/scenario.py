"""Replays a synthetic workload's events with the oracle pieces.

A workload (duck-typed: see workloads.gen.Workload) lists admissions, forks
and history appends; then one decode step in which every batch sequence
appends one token (block copies first, then the append) and attends over its
whole context. This mirrors the engine loop of cs2680 Lecture 10, §10.5
(allocate blocks to grow, run the step, append the emitted tokens), reduced
to one attention layer.
"""
from __future__ import annotations

import numpy as np

from . import cache_ops, paged_attention
from .block_manager import BlockManager


def _apply_events(w, bm, k_pool=None, v_pool=None):
    history = []
    for ei, ev in enumerate(w.events):
        kind = ev[0]
        if kind == "admit":
            _, prompt_len, max_new, group, prefix_len = ev
            bm.admit(prompt_len, max_new, group, prefix_len)
        elif kind == "fork":
            bm.fork(ev[1], ev[2])
        elif kind == "history":
            counts = ev[1]
            ids = sorted(counts)
            steps = max(counts.values()) if counts else 0
            for t in range(steps):
                batch = [s for s in ids if counts[s] > t]
                slots, pairs = bm.prepare_append(batch)
                history.append((batch, slots, pairs))
                if k_pool is not None:
                    cache_ops.copy_blocks(k_pool, v_pool, pairs)
                    k, v = w.history_inputs(ei, t, len(batch))
                    cache_ops.append_kv(k_pool, v_pool, k, v, slots)
        else:
            raise ValueError(f"unknown event {kind}")
    return history


def padded_tables(bm, seq_ids):
    width = max(len(bm.table(s)) for s in seq_ids)
    tables = np.full((len(seq_ids), width), -1, dtype=np.int32)
    for i, s in enumerate(seq_ids):
        t = bm.table(s)
        tables[i, : len(t)] = t
    return tables


def replay(w, attend: bool = True):
    """Full replay on a materialised pool. Returns a dict with the block
    manager, the history bookkeeping, the step's slots / pairs, the batch's
    block tables and context lengths, the pools after the step and (if
    `attend`) the float64 attention output [B, Hq, D]."""
    bm = BlockManager(w.pool_blocks, w.block_tokens, w.free_order)
    k_pool, v_pool = w.pool("k"), w.pool("v")
    history = _apply_events(w, bm, k_pool, v_pool)
    slots, pairs = bm.prepare_append(w.batch)
    cache_ops.copy_blocks(k_pool, v_pool, pairs)
    q, k_new, v_new = w.step_inputs()
    cache_ops.append_kv(k_pool, v_pool, k_new, v_new, slots)
    tables = padded_tables(bm, w.batch)
    ctx = np.array([bm.context_len(s) for s in w.batch], dtype=np.int64)
    res = dict(bm=bm, history=history, slots=slots, pairs=pairs, tables=tables,
               ctx=ctx, q=q, k_pool=k_pool, v_pool=v_pool)
    if attend:
        res["out"] = paged_attention.paged_decode_attention(
            q, k_pool, v_pool, tables, ctx, w.scale)
    return res


def replay_sampled(w, sample_rows):
    """Attention for the batch rows in `sample_rows` only, regenerating just
    the pool blocks those rows read. For workloads without history events
    (every token before the step is pool content). Returns (out_rows float64
    [len(sample_rows), Hq, D], the full-replay bookkeeping dict without pools)."""
    if any(ev[0] == "history" for ev in w.events):
        raise ValueError("sampled replay needs a workload without history appends")
    bm = BlockManager(w.pool_blocks, w.block_tokens, w.free_order)
    _apply_events(w, bm)
    slots, pairs = bm.prepare_append(w.batch)
    q, k_new, v_new = w.step_inputs()
    tables = padded_tables(bm, w.batch)
    ctx = np.array([bm.context_len(s) for s in w.batch], dtype=np.int64)
    rows = [int(r) for r in sample_rows]
    # physical blocks the sampled rows read, plus sources copied into them
    need = set()
    for r in rows:
        need.update(int(b) for b in tables[r, : -(-int(ctx[r]) // w.block_tokens)])
    need.update(s for s, d in pairs if d in need)
    need = sorted(need)
    remap = {b: i for i, b in enumerate(need)}
    k_loc = w.pool_blocks_at("k", need)
    v_loc = w.pool_blocks_at("v", need)
    loc_pairs = [(remap[s], remap[d]) for s, d in pairs if d in remap]
    cache_ops.copy_blocks(k_loc, v_loc, loc_pairs)
    b = w.block_tokens
    loc_slots = []
    for s in slots:
        blk = s // b
        loc_slots.append(remap[blk] * b + s % b if blk in remap else -1)
    cache_ops.append_kv(k_loc, v_loc, k_new, v_new, loc_slots)
    loc_tables = np.full((len(rows), tables.shape[1]), -1, dtype=np.int32)
    for i, r in enumerate(rows):
        n = -(-int(ctx[r]) // b)
        loc_tables[i, :n] = [remap[int(x)] for x in tables[r, :n]]
    out = paged_attention.paged_decode_attention(
        q[rows], k_loc, v_loc, loc_tables, ctx[rows], w.scale)
    return out, dict(bm=bm, slots=slots, pairs=pairs, tables=tables, ctx=ctx, q=q)
