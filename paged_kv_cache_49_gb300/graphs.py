"""Decode steps replayed from CUDA graphs captured per batch-size bucket.

"The inference server": because attention takes a block table and a length
tensor, both fixed-shape, the decode step's arguments stop changing shape as
sequences grow; only the batch size varies, and it is handled by bucketing:
capture a graph per bucket (1, 2, 4, 8, ...), pad the running batch up to the
next bucket, copy the block tables and lengths into the captured input
buffers, and replay. Padding rows carry slot -1 (the append writes nothing)
and context length 0 (a zero output row), so they cost almost nothing.

Copy-on-write pairs vary in number from step to step and are rare (a shared
partial block is copied once per sharer), so a step that has any launches the
block copy on the same stream just before the replay; the captured graph
itself is append + attention.
"""
from __future__ import annotations

import torch

from . import _native as nat
from .engine import PagedKVEngine, bf16_from_bits


def default_buckets(max_batch: int) -> list[int]:
    b, out = 1, []
    while b < max_batch:
        out.append(b)
        b *= 2
    out.append(max_batch)
    return out


class _Bucket:
    def __init__(self, eng: PagedKVEngine, size: int, width: int):
        dev = eng.device
        hq, hkv, d = eng.num_q_heads, eng.num_kv_heads, eng.head_dim
        self.size = size
        self.q = torch.zeros((size, hq, d), dtype=torch.bfloat16, device=dev)
        self.k = torch.zeros((size, hkv, d), dtype=torch.bfloat16, device=dev)
        self.v = torch.zeros((size, hkv, d), dtype=torch.bfloat16, device=dev)
        self.slots = torch.full((size,), -1, dtype=torch.int64, device=dev)
        self.tables = torch.full((size, width), -1, dtype=torch.int32, device=dev)
        self.ctx = torch.zeros((size,), dtype=torch.int32, device=dev)
        self.out = torch.zeros((size, hq, d), dtype=torch.bfloat16, device=dev)
        self.no_pairs = torch.zeros((0, 2), dtype=torch.int32, device=dev)
        self.ws = nat.AttentionWorkspace(size, hkv, device=dev)
        # pinned staging for the host-side inputs of a step
        self.h_slots = torch.full((size,), -1, dtype=torch.int64).pin_memory()
        self.h_tables = torch.full((size, width), -1, dtype=torch.int32).pin_memory()
        self.h_ctx = torch.zeros((size,), dtype=torch.int32).pin_memory()
        self.staged = torch.cuda.Event()  # the last copies out of the staging buffers have run
        self.graph = None


class GraphedDecoder:
    """Replays captured decode steps for an engine's pool and block manager."""

    def __init__(self, eng: PagedKVEngine, max_batch: int, max_blocks_per_seq: int, scale: float,
                 buckets=None, num_ctas: int = 0):
        self.eng, self.scale, self.num_ctas = eng, float(scale), num_ctas
        self.width = max_blocks_per_seq
        self.buckets = {b: _Bucket(eng, b, max_blocks_per_seq) for b in (buckets or default_buckets(max_batch))}
        for b in self.buckets.values():
            self._capture(b)

    def _launch(self, b: _Bucket):
        nat.decode_step(b.q, b.k, b.v, b.slots, b.no_pairs, self.eng.k_cache, self.eng.v_cache, b.tables, b.ctx,
                        self.scale, b.out, b.ws, self.eng.error, self.num_ctas)

    def _capture(self, b: _Bucket):
        # All-padding inputs: the warm-up launch writes nothing to the pool.
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self._launch(b)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        b.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(b.graph):
            self._launch(b)

    def bucket_for(self, n: int) -> _Bucket:
        for size in sorted(self.buckets):
            if size >= n:
                return self.buckets[size]
        raise ValueError(f"batch of {n} exceeds the largest bucket {max(self.buckets)}")

    def step(self, seq_ids, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor):
        """One decode step for the listed sequences: q [n, Hq, D], k, v
        [n, Hkv, D] (bf16, on the device or pinned host memory). Returns
        (out view [n, Hq, D], slots, pairs)."""
        n = len(seq_ids)
        b = self.bucket_for(n)
        b.staged.synchronize()  # the previous step's copies have read the staging buffers
        slots, pairs = self.eng.bm.prepare_append(list(seq_ids))
        tables, ctx = self.eng.bm.batch_tables(list(seq_ids), self.width)
        b.h_slots[:n] = torch.tensor(slots, dtype=torch.int64)
        b.h_slots[n:] = -1
        b.h_tables[:n] = tables
        b.h_tables[n:] = -1
        b.h_ctx[:n] = ctx
        b.h_ctx[n:] = 0
        b.slots.copy_(b.h_slots, non_blocking=True)
        b.tables.copy_(b.h_tables, non_blocking=True)
        b.ctx.copy_(b.h_ctx, non_blocking=True)
        b.q[:n].copy_(q, non_blocking=True)
        b.k[:n].copy_(k, non_blocking=True)
        b.v[:n].copy_(v, non_blocking=True)
        b.staged.record()
        if pairs:
            pt = torch.tensor(pairs, dtype=torch.int32).to(self.eng.device, non_blocking=True)
            nat.block_copy(self.eng.k_cache, self.eng.v_cache, pt, self.eng.error)
        b.graph.replay()
        return b.out[:n], slots, pairs

    def step_bits(self, seq_ids, q_bits, k_bits, v_bits):
        """step() from bf16 bit patterns held in numpy arrays."""
        return self.step(seq_ids, bf16_from_bits(q_bits), bf16_from_bits(k_bits), bf16_from_bits(v_bits))
