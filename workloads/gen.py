"""Seeded synthetic workloads for paged decode attention.

Everything here is a random draw or a shape. A workload is a list of
block-manager events (admit / fork / history appends) plus deterministic
content generators; the oracle side and the CUDA side each replay the events
with their own code.

Values are N(0, 1) drawn by inverse-transform sampling: a 16-bit uniform
index picks one of 65,536 equal-probability normal quantiles, stored as bf16
bit patterns. Pool content is generated in chunks of CHUNK_BLOCKS physical
blocks, each chunk from its own seed, so that a caller can regenerate any
block range without materialising the whole pool.

The shapes follow the pages' geometries: Llama-3-8B (32 q / 8 kv heads,
d_h = 128) and Llama-3.3-70B (64 q / 8 kv heads, d_h = 128) in BF16 with
16-token blocks ("The inference server"; "KV cache systems", kv bytes/token
equation); the prefix-sharing admission case of "Reserve the page a request
has not written yet" (2,048-token prefix, 257-token suffix, 256-page pool);
and parallel-sampling fan-out (cs2680 Lecture 10, §10.4).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from statistics import NormalDist

import numpy as np

BLOCK_TOKENS = 16
CHUNK_BLOCKS = 64

# Distinct seed-sequence tags per stream, so streams never overlap.
_TAG_POOL_K, _TAG_POOL_V, _TAG_STEP, _TAG_HIST, _TAG_PARAMS = 11, 12, 13, 14, 15


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def _normal_table() -> np.ndarray:
    nd = NormalDist()
    p = (np.arange(65536, dtype=np.float64) + 0.5) / 65536.0
    vals = np.array([nd.inv_cdf(float(pi)) for pi in p], dtype=np.float32)
    return bf16_bits(vals)


_NORMAL_BF16: np.ndarray | None = None


def randn_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0, 1) samples as bf16 bit patterns (uint16) of the given shape."""
    global _NORMAL_BF16
    if _NORMAL_BF16 is None:
        _NORMAL_BF16 = _normal_table()
    idx = rng.integers(0, 65536, size=shape, dtype=np.uint16)
    return _NORMAL_BF16[idx]


def _rng(seed: int, *tags: int) -> np.random.Generator:
    return np.random.default_rng([seed, *tags])


@dataclass
class Workload:
    """One synthetic decode workload.

    events: ordered list of
      ("admit", prompt_len, max_new, group, prefix_len)  -> next sequence id
      ("fork", parent_seq, n)                            -> n next sequence ids
      ("history", {seq_id: n_tokens})                    -> n_tokens appends per
          sequence before the measured step; step t batches, in ascending id
          order, every sequence with n_tokens > t.
    batch: sequence ids of the measured decode step, in batch order (each
      sequence appends one token, then attends over its whole context).
    """

    name: str
    description: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    pool_blocks: int
    events: list = field(default_factory=list)
    batch: list = field(default_factory=list)
    free_order: np.ndarray | None = None
    pool_fill: str = "randn"  # "randn" or "nan" (every slot NaN until appended)
    block_tokens: int = BLOCK_TOKENS

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def batch_size(self) -> int:
        return len(self.batch)

    # ---- content -------------------------------------------------------
    def block_shape(self):
        return (self.num_kv_heads, self.block_tokens, self.head_dim)

    def pool_chunk(self, which: str, chunk: int) -> np.ndarray:
        """Blocks [chunk*CHUNK_BLOCKS, ...) of the K ('k') or V ('v') pool."""
        lo = chunk * CHUNK_BLOCKS
        hi = min(self.pool_blocks, lo + CHUNK_BLOCKS)
        shape = (hi - lo,) + self.block_shape()
        if self.pool_fill == "nan":
            return np.full(shape, 0x7FC0, dtype=np.uint16)
        tag = _TAG_POOL_K if which == "k" else _TAG_POOL_V
        return randn_bf16(_rng(self.seed, tag, chunk), shape)

    def pool_blocks_range(self, which: str, lo: int, hi: int) -> np.ndarray:
        out = np.empty((hi - lo,) + self.block_shape(), dtype=np.uint16)
        c0, c1 = lo // CHUNK_BLOCKS, (hi - 1) // CHUNK_BLOCKS
        for c in range(c0, c1 + 1):
            blk = self.pool_chunk(which, c)
            a = max(lo, c * CHUNK_BLOCKS)
            b = min(hi, c * CHUNK_BLOCKS + blk.shape[0])
            out[a - lo : b - lo] = blk[a - c * CHUNK_BLOCKS : b - c * CHUNK_BLOCKS]
        return out

    def pool(self, which: str) -> np.ndarray:
        return self.pool_blocks_range(which, 0, self.pool_blocks)

    def pool_blocks_at(self, which: str, ids) -> np.ndarray:
        """Initial content of the listed physical blocks, generating each
        chunk once."""
        ids = [int(i) for i in ids]
        out = np.empty((len(ids),) + self.block_shape(), dtype=np.uint16)
        by_chunk: dict[int, list[int]] = {}
        for pos, b in enumerate(ids):
            by_chunk.setdefault(b // CHUNK_BLOCKS, []).append(pos)
        for c, positions in by_chunk.items():
            blk = self.pool_chunk(which, c)
            for pos in positions:
                out[pos] = blk[ids[pos] - c * CHUNK_BLOCKS]
        return out

    def step_inputs(self):
        """(q [B, Hq, D], k_new [B, Hkv, D], v_new [B, Hkv, D]) as bf16 bits."""
        r = _rng(self.seed, _TAG_STEP)
        B, D = self.batch_size, self.head_dim
        q = randn_bf16(r, (B, self.num_q_heads, D))
        k = randn_bf16(r, (B, self.num_kv_heads, D))
        v = randn_bf16(r, (B, self.num_kv_heads, D))
        return q, k, v

    def history_inputs(self, event_index: int, t: int, n: int):
        """(k [n, Hkv, D], v [n, Hkv, D]) for history step t of one event."""
        r = _rng(self.seed, _TAG_HIST, event_index, t)
        shape = (n, self.num_kv_heads, self.head_dim)
        return randn_bf16(r, shape), randn_bf16(r, shape)


def _lognormal_lengths(rng, n, median, sigma, lo, hi):
    x = rng.lognormal(mean=math.log(median), sigma=sigma, size=n)
    return np.clip(np.rint(x), lo, hi).astype(np.int64)


def _pool_bound(token_counts, slack=1.1, block_tokens=BLOCK_TOKENS):
    """Pool size (blocks) comfortably above the pages the requests reserve."""
    tokens = int(np.sum(token_counts))
    return int(math.ceil(slack * (tokens / block_tokens + len(token_counts))))


def _decode_batch(name, desc, seed, hq, hkv, ctx, pool_blocks=None, fill="randn", block_tokens=BLOCK_TOKENS):
    """Every sequence holds ctx-1 tokens and appends its ctx-th in the step."""
    ctx = [int(c) for c in ctx]
    events = [("admit", c - 1, 1, -1, 0) for c in ctx]
    if pool_blocks is None:
        pool_blocks = _pool_bound(ctx, block_tokens=block_tokens)
    w = Workload(name, desc, seed, hq, hkv, 128, pool_blocks, events, list(range(len(ctx))),
                 block_tokens=block_tokens)
    w.free_order = _rng(seed, _TAG_PARAMS, 1).permutation(pool_blocks).astype(np.int32)
    w.pool_fill = fill
    return w


def tiny(seed: int = 0, block_tokens: int = BLOCK_TOKENS) -> Workload:
    return _decode_batch(
        "tiny", "batch 4, ctx {1,16,17,203}, 32 q / 8 kv heads, d_h 128, 64-block permuted pool",
        seed, 32, 8, [1, 16, 17, 203], pool_blocks=64, block_tokens=block_tokens)


def tiny_nan(seed: int = 0) -> Workload:
    """Tiny batch whose pool starts all-NaN: every valid token is written by
    append, so any read of an unwritten slot shows up as a non-finite output."""
    ctx = [1, 16, 17, 203]
    events = [("admit", 0, c, -1, 0) for c in ctx]
    hist = {i: c - 1 for i, c in enumerate(ctx) if c > 1}
    events.append(("history", hist))
    w = Workload("tiny_nan", "tiny batch, NaN-filled pool, content written by appends",
                 seed, 32, 8, 128, 64, events, list(range(4)))
    w.free_order = _rng(seed, _TAG_PARAMS, 1).permutation(64).astype(np.int32)
    w.pool_fill = "nan"
    return w


def llama3_8b(seed: int = 0, batch: int = 64, block_tokens: int = BLOCK_TOKENS) -> Workload:
    r = _rng(seed, _TAG_PARAMS, 0)
    ctx = _lognormal_lengths(r, batch, 1024, 1.0, 1, 8192)
    return _decode_batch(
        "llama3_8b_b64", "Llama-3-8B geometry, batch 64, lognormal(1024, 1.0) ctx in [1, 8192]",
        seed, 32, 8, ctx, block_tokens=block_tokens)


def llama33_70b(seed: int = 0, batch: int = 256, block_tokens: int = BLOCK_TOKENS) -> Workload:
    r = _rng(seed, _TAG_PARAMS, 0)
    ctx = _lognormal_lengths(r, batch, 4096, 1.2, 16, 131072)
    ctx[:4] = 131072
    return _decode_batch(
        "llama33_70b_b256",
        "Llama-3.3-70B geometry, batch 256, lognormal(4096, 1.2) ctx in [16, 131072], seqs 0-3 at 131072",
        seed, 64, 8, ctx, block_tokens=block_tokens)


def prefix_admission(seed: int = 0) -> Workload:
    """Seven requests share a 2,048-token prefix (128 pages) in a 256-page pool,
    each reserving 257 output tokens; each has produced a seeded number of
    suffix tokens. Request 0 is at suffix position 200 and is then forked once,
    so that its partial last block is shared and the next write copies it."""
    r = _rng(seed, _TAG_PARAMS, 0)
    produced = r.integers(1, 257, size=7)  # suffix tokens already written (1..256)
    produced[0] = 200
    events = [("admit", 2048, 257, 0, 2048) for _ in range(7)]
    events.append(("history", {i: int(produced[i]) for i in range(7)}))
    events.append(("fork", 0, 1))
    w = Workload("prefix_admission", "7 requests x (2048 shared + 257 private), 256-page pool, one CoW fork",
                 seed, 32, 8, 128, 256, events, list(range(8)))
    w.free_order = _rng(seed, _TAG_PARAMS, 1).permutation(256).astype(np.int32)
    return w


def fanout(seed: int = 0, prompts: int = 16, samples: int = 8) -> Workload:
    """16 prompts x 8 samples: each prompt's blocks are shared by its samples
    (the admitted request plus 7 forks); each sample has produced a seeded
    number of private output tokens in [1, 512]."""
    r = _rng(seed, _TAG_PARAMS, 0)
    plen = r.integers(512, 4097, size=prompts)
    outs = r.integers(1, 513, size=prompts * samples)
    events, batch, hist = [], [], {}
    next_id = 0
    for p in range(prompts):
        events.append(("admit", int(plen[p]), 512, -1, 0))
        parent = next_id
        next_id += 1
        events.append(("fork", parent, samples - 1))
        ids = [parent] + list(range(next_id, next_id + samples - 1))
        next_id += samples - 1
        batch.extend(ids)
    for i, sid in enumerate(batch):
        if outs[i] > 1:
            hist[sid] = int(outs[i]) - 1
    events.append(("history", hist))
    # prompt stored once, each sample's 512-token allowance plus one block of slack
    reserved = [int(plen[p]) + samples * (512 + BLOCK_TOKENS) for p in range(prompts)]
    w = Workload("fanout", "16 prompts x 8 samples, prompts U[512,4096] shared, outputs U[1,512] private",
                 seed, 32, 8, 128, _pool_bound(reserved), events, batch)
    w.free_order = _rng(seed, _TAG_PARAMS, 1).permutation(w.pool_blocks).astype(np.int32)
    return w


def heads(seed: int = 0, hq: int = 8, hkv: int = 8) -> Workload:
    """Edge shapes of the GQA mapping: MHA (G = 1), G = 2, MQA (one KV head),
    on a small ragged batch that spans several blocks and a partial tail."""
    return _decode_batch(f"heads_{hq}_{hkv}", f"batch 6, ctx mix, {hq} q / {hkv} kv heads", seed, hq, hkv,
                         [1, 15, 16, 33, 200, 517])


def long_single(seed: int = 0) -> Workload:
    """One 131,072-token sequence with the 70B geometry: every CTA holds a
    piece of the same (sequence, KV head) runs, so the merge spans many CTAs."""
    return _decode_batch("long_single", "batch 1, ctx 131072, 64 q / 8 kv heads", seed, 64, 8, [131072])


def many_short(seed: int = 0) -> Workload:
    """The largest batch the kernel takes (4,096 sequences), 1..40 tokens each:
    thousands of short runs and pieces per CTA."""
    r = _rng(seed, _TAG_PARAMS, 0)
    ctx = r.integers(1, 41, size=4096)
    return _decode_batch("many_short", "batch 4096, ctx U[1, 40], 32 q / 8 kv heads", seed, 32, 8, ctx)


def large_batch(seed: int = 0, batch: int = 4096) -> Workload:
    """A large decode batch at moderate contexts (lognormal, median 256 tokens,
    clipped to [16, 2,048]): bandwidth-bound like the 64-sequence batch, but
    with thousands of (sequence, KV head) runs per launch."""
    r = _rng(seed, _TAG_PARAMS, 0)
    ctx = _lognormal_lengths(r, batch, 256, 0.5, 16, 2048)
    return _decode_batch(f"large_batch_{batch}", f"batch {batch}, lognormal(256, 0.5) ctx in [16, 2048], 32 q / 8 kv heads",
                         seed, 32, 8, ctx)


WORKLOADS = {
    "heads_8_8": lambda seed=0: heads(seed, 8, 8),
    "heads_16_8": lambda seed=0: heads(seed, 16, 8),
    "heads_8_1": lambda seed=0: heads(seed, 8, 1),
    "heads_64_8": lambda seed=0: heads(seed, 64, 8),
    "long_single": long_single,
    "many_short": many_short,
    "large_batch_4096": lambda seed=0: large_batch(seed, 4096),
    "large_batch_2048": lambda seed=0: large_batch(seed, 2048),
    "tiny": tiny,
    "tiny_nan": tiny_nan,
    "llama3_8b_b64": llama3_8b,
    "prefix_admission": prefix_admission,
    "fanout": fanout,
    "llama33_70b_b256": llama33_70b,
}


def make_workload(name: str, seed: int = 0, **kw) -> Workload:
    return WORKLOADS[name](seed=seed, **kw)
