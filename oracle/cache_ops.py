"""Slot arithmetic, KV append and block copy, restated.

cs2680 Lecture 10, §10.3: a sequence's logical block i maps to whichever
physical block its table names; growing by one token writes one slot of the
last block (or of a newly acquired block). "KV cache systems", copy-on-write
paragraph: the first writer of a shared block gets a copy, so only the
divergent suffix takes new memory.

slot = physical_block * b + (position mod b), with physical_block =
table[position // b]; slot < 0 marks a padding row that writes nothing.
"""
from __future__ import annotations

import numpy as np


def slot_of(table_row, position: int, block_tokens: int = 16) -> int:
    return int(table_row[position // block_tokens]) * block_tokens + position % block_tokens


def append_kv(k_cache, v_cache, k_new, v_new, slot_mapping) -> None:
    """In place: row i of k_new / v_new [T, Hkv, D] goes to slot slot_mapping[i]."""
    b = k_cache.shape[2]
    for i, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0:
            continue
        blk, row = divmod(slot, b)
        k_cache[blk, :, row, :] = k_new[i]
        v_cache[blk, :, row, :] = v_new[i]


def copy_blocks(k_cache, v_cache, pairs) -> None:
    """In place: for each (src, dst), physical block dst becomes a copy of src
    (all KV heads, all rows). Sources are read before any destination is
    written, so the result does not depend on pair order."""
    pairs = [(int(s), int(d)) for s, d in pairs]
    if not pairs:
        return
    src = np.array([p[0] for p in pairs])
    dst = np.array([p[1] for p in pairs])
    k_src, v_src = k_cache[src].copy(), v_cache[src].copy()
    k_cache[dst] = k_src
    v_cache[dst] = v_src
