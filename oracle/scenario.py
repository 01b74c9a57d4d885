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


def sampled_inputs(w, sample_rows):
    """The decode step's inputs restricted to the batch rows in `sample_rows`,
    regenerating just the pool blocks those rows read (for workloads without
    history events: every token before the step is pool content). Returns a
    dict: q, k_new, v_new (the sampled rows'), k_pool / v_pool (the needed
    blocks before the step's copies and appends, renumbered), pairs and slots
    (the step's copies and the sampled rows' appends in that numbering, -1
    for an append outside it), tables and ctx (the sampled rows'),
    loc_slots_all (every batch row's append in that numbering) and the full
    batch's bookkeeping (bm, all_slots, all_pairs, all_tables, all_ctx, all_q,
    all_k_new, all_v_new)."""
    if any(ev[0] == "history" for ev in w.events):
        raise ValueError("sampled replay needs a workload without history appends")
    bm = BlockManager(w.pool_blocks, w.block_tokens, w.free_order)
    _apply_events(w, bm)
    slots, pairs = bm.prepare_append(w.batch)
    q, k_new, v_new = w.step_inputs()
    tables = padded_tables(bm, w.batch)
    ctx = np.array([bm.context_len(s) for s in w.batch], dtype=np.int64)
    rows = [int(r) for r in sample_rows]
    b = w.block_tokens
    # physical blocks the sampled rows read, plus sources copied into them
    need = set()
    for r in rows:
        need.update(int(x) for x in tables[r, : -(-int(ctx[r]) // b)])
    need.update(s for s, d in pairs if d in need)
    need = sorted(need)
    remap = {blk: i for i, blk in enumerate(need)}
    loc_pairs = [(remap[s], remap[d]) for s, d in pairs if d in remap]
    # every batch row's append in the new numbering (-1 outside it)
    loc_slots_all = []
    for sl in slots:
        blk = sl // b
        loc_slots_all.append(remap[blk] * b + sl % b if blk in remap else -1)
    loc_tables = np.full((len(rows), tables.shape[1]), -1, dtype=np.int32)
    for i, r in enumerate(rows):
        n = -(-int(ctx[r]) // b)
        loc_tables[i, :n] = [remap[int(x)] for x in tables[r, :n]]
    return dict(q=q[rows], k_new=k_new[rows], v_new=v_new[rows],
                k_pool=w.pool_blocks_at("k", need), v_pool=w.pool_blocks_at("v", need),
                pairs=loc_pairs, slots=[loc_slots_all[r] for r in rows], tables=loc_tables, ctx=ctx[rows],
                loc_slots_all=loc_slots_all, all_k_new=k_new, all_v_new=v_new,
                bm=bm, all_slots=slots, all_pairs=pairs, all_tables=tables, all_ctx=ctx, all_q=q)


def replay_sampled(w, sample_rows):
    """Attention for the batch rows in `sample_rows` only, regenerating just
    the pool blocks those rows read. For workloads without history appends
    (every token before the step is pool content). Returns (out_rows float64
    [len(sample_rows), Hq, D], the full-replay bookkeeping dict without pools)."""
    inp = sampled_inputs(w, sample_rows)
    k_loc, v_loc = inp["k_pool"], inp["v_pool"]
    cache_ops.copy_blocks(k_loc, v_loc, inp["pairs"])
    cache_ops.append_kv(k_loc, v_loc, inp["all_k_new"], inp["all_v_new"], inp["loc_slots_all"])
    out = paged_attention.paged_decode_attention(
        inp["q"], k_loc, v_loc, inp["tables"], inp["ctx"], w.scale)
    return out, dict(bm=inp["bm"], slots=inp["all_slots"], pairs=inp["all_pairs"], tables=inp["all_tables"],
                     ctx=inp["all_ctx"], q=inp["all_q"])
