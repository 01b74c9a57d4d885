"""One attention layer's paged KV cache on one GPU.

The pool is allocated once as two device arrays [num_blocks, Hkv, 16, D]
("The inference server": the KV cache is one arena allocated at start-up,
managed by block tables, with no allocator on the hot path). The C++ block
manager owns the tables; a decode step is host bookkeeping (slots and
copy-on-write pairs from pkv_bm_prepare_append, cs2680 Lecture 10, §10.5's
"allocate blocks to grow") followed by three launches on one stream: block
copy, append, attention.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import _native as nat


def bf16_from_bits(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns -> CPU bf16 tensor sharing no arithmetic."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def bits_from_bf16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def shared_prefix_groups(tables, context_lens, block_tokens: int = nat.BLOCK_TOKENS, min_members: int = 2):
    """Groups of a batch's sequences that share leading blocks, for cascade
    attention: sequences whose tables start with the same block form a group
    (of at least min_members); its shared length is the longest table prefix
    all members agree on, limited to the complete blocks of the shortest
    member (a shared tile must be whole for every sharer). Host arithmetic on
    the batch's block tables; returns [(member indices, shared blocks)]."""
    tables = np.asarray(tables)
    ctx = np.asarray(context_lens, dtype=np.int64)
    by_first = {}
    for s in range(len(ctx)):
        if ctx[s] >= block_tokens:
            by_first.setdefault(int(tables[s, 0]), []).append(s)
    groups = []
    for members in by_first.values():
        if len(members) < min_members:
            continue
        limit = int(min(ctx[m] // block_tokens for m in members))
        rows = tables[members, :limit]
        agree = np.all(rows == rows[0], axis=0)
        shared = limit if agree.all() else int(np.argmin(agree))
        if shared >= 1:
            groups.append((members, shared))
    return groups


# Below this many K/V bytes saved, the cascade's extra launches cost more than
# the shared reads they avoid (measured: a 7-request group sharing 128 blocks,
# 59 MB saved, ran slower than the plain kernel; 16 prompts x 8 samples,
# 1.06 GB saved, ran 2.3x faster).
CASCADE_MIN_SAVED_BYTES = 128 << 20


def cascade_saved_bytes(groups, num_kv_heads: int, block_tokens: int = nat.BLOCK_TOKENS, head_dim: int = 128) -> int:
    """K and V bytes cascade attention does not read: every sharer but one of
    each group skips the group's shared blocks."""
    per_block = num_kv_heads * block_tokens * head_dim * 2 * 2
    return sum((len(m) - 1) * sh * per_block for m, sh in groups)


@dataclass
class StepBuffers:
    """Device inputs and output of one decode step (shapes fixed per batch)."""
    seq_ids: list
    slots: torch.Tensor       # int64 [B]
    pairs: torch.Tensor       # int32 [n, 2]
    tables: torch.Tensor      # int32 [B, W]
    ctx: torch.Tensor         # int32 [B]
    q: torch.Tensor           # bf16 [B, Hq, D]
    k: torch.Tensor           # bf16 [B, Hkv, D]
    v: torch.Tensor           # bf16 [B, Hkv, D]
    out: torch.Tensor         # bf16 [B, Hq, D]
    workspace: nat.AttentionWorkspace

    @property
    def num_pairs(self) -> int:
        return int(self.pairs.shape[0])


class PagedKVEngine:
    def __init__(self, num_blocks: int, num_q_heads: int, num_kv_heads: int, head_dim: int = 128,
                 device="cuda", free_order=None, block_tokens: int = nat.BLOCK_TOKENS, incremental: bool = False,
                 watermark: int = 0, prefix_cache: bool = False):
        self.num_blocks, self.num_q_heads, self.num_kv_heads, self.head_dim = (
            num_blocks, num_q_heads, num_kv_heads, head_dim)
        self.block_tokens = block_tokens
        self.device = torch.device(device)
        shape = (num_blocks, num_kv_heads, block_tokens, head_dim)
        self.k_cache = torch.empty(shape, dtype=torch.bfloat16, device=self.device)
        self.v_cache = torch.empty(shape, dtype=torch.bfloat16, device=self.device)
        self.bm = nat.BlockManager(num_blocks, block_tokens, free_order, incremental=incremental,
                                   watermark=watermark, prefix_cache=prefix_cache)
        self.error = nat.new_error_word(self.device)

    # ---- pool content ----------------------------------------------------
    def load_pool(self, k_bits: np.ndarray, v_bits: np.ndarray, lo: int = 0) -> None:
        n = k_bits.shape[0]
        self.k_cache[lo : lo + n].copy_(bf16_from_bits(k_bits))
        self.v_cache[lo : lo + n].copy_(bf16_from_bits(v_bits))

    def load_workload_pool(self, w, chunk_blocks: int = 4096) -> None:
        for lo in range(0, w.pool_blocks, chunk_blocks):
            hi = min(w.pool_blocks, lo + chunk_blocks)
            self.load_pool(w.pool_blocks_range("k", lo, hi), w.pool_blocks_range("v", lo, hi), lo)

    # ---- host bookkeeping + device launches ---------------------------------
    def append_tokens(self, seq_ids, k: torch.Tensor, v: torch.Tensor, stream=None):
        """Append one token per sequence (k, v: [B, Hkv, D] bf16 on device);
        returns (slots, pairs) as the block manager decided them."""
        slots, pairs = self.bm.prepare_append(list(seq_ids))
        if pairs:
            pt = torch.tensor(pairs, dtype=torch.int32).to(self.device, non_blocking=True)
            nat.block_copy(self.k_cache, self.v_cache, pt, self.error, stream)
        st = torch.tensor(slots, dtype=torch.int64).to(self.device, non_blocking=True)
        nat.append(k, v, st, self.k_cache, self.v_cache, self.error, stream)
        return slots, pairs

    def write_positions(self, seq_id: int, first: int, k: torch.Tensor, v: torch.Tensor, stream=None):
        """Write the KV of token positions [first, first + n) of one sequence
        (k, v: [n, Hkv, D] bf16 on device) -- a prefill, or the recompute of a
        resumed sequence -- with the append kernel; returns the slots."""
        slots = self.bm.slots(seq_id, first, int(k.shape[0]))
        st = torch.tensor(slots, dtype=torch.int64).to(self.device, non_blocking=True)
        nat.append(k, v, st, self.k_cache, self.v_cache, self.error, stream)
        return slots

    def replay_events(self, w, with_content: bool = True):
        """Apply a workload's admit / fork / history events; history appends
        write the workload's history K/V when with_content is set."""
        history = []
        for ei, ev in enumerate(w.events):
            if ev[0] == "admit":
                self.bm.admit(ev[1], ev[2], ev[3], ev[4])
            elif ev[0] == "fork":
                self.bm.fork(ev[1], ev[2])
            elif ev[0] == "history":
                counts = ev[1]
                ids = sorted(counts)
                for t in range(max(counts.values()) if counts else 0):
                    batch = [s for s in ids if counts[s] > t]
                    if with_content:
                        kb, vb = w.history_inputs(ei, t, len(batch))
                        k = bf16_from_bits(kb).to(self.device)
                        v = bf16_from_bits(vb).to(self.device)
                        slots, pairs = self.append_tokens(batch, k, v)
                    else:
                        slots, pairs = self.bm.prepare_append(batch)
                    history.append((batch, slots, pairs))
            else:
                raise ValueError(f"unknown event {ev[0]}")
        return history

    def prepare_step(self, seq_ids, q_bits, k_bits, v_bits, width: int | None = None) -> StepBuffers:
        """Host bookkeeping of one decode step (each sequence appends one
        token) and its device inputs; the step itself is run_step."""
        seq_ids = list(seq_ids)
        slots, pairs = self.bm.prepare_append(seq_ids)
        if width is None:
            width = max(len(self.bm.table(s)) for s in seq_ids)
        tables, ctx = self.bm.batch_tables(seq_ids, width)
        dev = self.device
        q = bf16_from_bits(q_bits).to(dev)
        return StepBuffers(
            seq_ids=seq_ids,
            slots=torch.tensor(slots, dtype=torch.int64).to(dev),
            pairs=torch.tensor(pairs, dtype=torch.int32).reshape(-1, 2).to(dev),
            tables=tables.to(dev), ctx=ctx.to(dev), q=q,
            k=bf16_from_bits(k_bits).to(dev), v=bf16_from_bits(v_bits).to(dev),
            out=torch.empty_like(q),
            workspace=nat.AttentionWorkspace(len(seq_ids), self.num_kv_heads, device=dev))

    def run_step(self, sb: StepBuffers, scale: float, num_ctas: int = 0, stream=None) -> torch.Tensor:
        """The device part of a decode step -- copy-on-write copies, append,
        attention -- as one library call (separate calls for block sizes
        other than 16). Idempotent for fixed inputs."""
        if self.block_tokens != nat.BLOCK_TOKENS:
            return self.run_step_separate(sb, scale, num_ctas, stream)
        return nat.decode_step(sb.q, sb.k, sb.v, sb.slots, sb.pairs, self.k_cache, self.v_cache, sb.tables,
                               sb.ctx, scale, sb.out, sb.workspace, self.error, num_ctas, stream)

    def run_step_separate(self, sb: StepBuffers, scale: float, num_ctas: int = 0, stream=None) -> torch.Tensor:
        """The same step as three separate library calls."""
        if sb.num_pairs:
            nat.block_copy(self.k_cache, self.v_cache, sb.pairs, self.error, stream)
        nat.append(sb.k, sb.v, sb.slots, self.k_cache, self.v_cache, self.error, stream)
        nat.attn_decode(sb.q, self.k_cache, self.v_cache, sb.tables, sb.ctx, scale, sb.out,
                        sb.workspace, num_ctas, stream)
        return sb.out

    def cascade_for(self, sb: StepBuffers, min_saved_bytes: int = CASCADE_MIN_SAVED_BYTES):
        """A cascade plan for the step's batch when its shared prefixes save
        enough reads to pay for the extra launches, else None."""
        if self.block_tokens != nat.BLOCK_TOKENS:
            return None
        groups = shared_prefix_groups(sb.tables.cpu().numpy(), sb.ctx.cpu().numpy())
        if not groups or cascade_saved_bytes(groups, self.num_kv_heads, head_dim=self.head_dim) < min_saved_bytes:
            return None
        return nat.Cascade(len(sb.seq_ids), self.num_q_heads, self.num_kv_heads, groups, device=self.device)

    def run_step_cascade(self, sb: StepBuffers, scale: float, cascade, stream=None) -> torch.Tensor:
        """run_step with the attention through a cascade plan (copy-on-write
        copies and the append first, as in run_step)."""
        if sb.num_pairs:
            nat.block_copy(self.k_cache, self.v_cache, sb.pairs, self.error, stream)
        nat.append(sb.k, sb.v, sb.slots, self.k_cache, self.v_cache, self.error, stream)
        return cascade.decode(sb.q, self.k_cache, self.v_cache, sb.tables, sb.ctx, scale, sb.out, stream)

    def read_errors(self, sb: StepBuffers | None = None) -> int:
        e = nat.read_device_error(self.error)
        if sb is not None:
            e |= sb.workspace.read_error()
        return e


class HostStep:
    """A decode step whose inputs and output live in host memory: one pinned
    packed input buffer (laid out by pkv_step_layout), its device staging
    buffer, and pinned output rows. run() is one pkv_decode_step_host call:
    a staging kernel reads the inputs across the host link, the step's
    kernels run, and the attention writes the output rows to host memory."""

    _DTYPES = {"q": torch.bfloat16, "k_new": torch.bfloat16, "v_new": torch.bfloat16, "slot_mapping": torch.int64,
               "block_tables": torch.int32, "context_lens": torch.int32, "src_dst_pairs": torch.int32}

    def __init__(self, eng: PagedKVEngine, num_seqs: int, width: int, max_pairs: int = 0):
        if eng.block_tokens != nat.BLOCK_TOKENS:
            raise ValueError("host-buffer steps use 16-token blocks")
        self.eng, self.num_seqs, self.width, self.max_pairs = eng, num_seqs, width, max_pairs
        hq, hkv, d = eng.num_q_heads, eng.num_kv_heads, eng.head_dim
        self.layout = nat.step_layout(num_seqs, hq, hkv, d, width, max_pairs)
        self.shapes = {"q": (num_seqs, hq, d), "k_new": (num_seqs, hkv, d), "v_new": (num_seqs, hkv, d),
                       "slot_mapping": (num_seqs,), "block_tables": (num_seqs, width),
                       "context_lens": (num_seqs,), "src_dst_pairs": (max_pairs, 2)}
        nbytes = self.layout["bytes"]
        self.host = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
        buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=eng.device)
        off = (-buf.data_ptr()) % 256
        self._staging_buf, self.staging = buf, buf[off: off + nbytes]
        self.out_dev = torch.empty((num_seqs, hq, d), dtype=torch.bfloat16, device=eng.device)
        self.out_host = torch.empty((num_seqs, hq, d), dtype=torch.bfloat16).pin_memory()
        self.workspace = nat.AttentionWorkspace(num_seqs, hkv, device=eng.device)
        self.num_pairs = 0

    def field(self, name: str, rows: int | None = None) -> torch.Tensor:
        """Typed view of one input inside the pinned packed buffer."""
        shape = list(self.shapes[name])
        if rows is not None:
            shape[0] = rows
        dt = self._DTYPES[name]
        n = int(np.prod(shape)) * torch.tensor([], dtype=dt).element_size()
        off = self.layout[name]
        return self.host[off: off + n].view(dt).view(shape)

    def pack(self, q, k, v, slots, tables, ctx, pairs=None) -> int:
        """Copy a step's inputs (CPU tensors) into the packed buffer; returns
        its size in bytes for this number of pairs."""
        self.field("q").copy_(q)
        self.field("k_new").copy_(k)
        self.field("v_new").copy_(v)
        self.field("slot_mapping").copy_(torch.as_tensor(slots, dtype=torch.int64))
        self.field("block_tables").copy_(tables)
        self.field("context_lens").copy_(ctx)
        n = 0 if pairs is None else int(len(pairs))
        if n > self.max_pairs:
            raise ValueError(f"{n} copy pairs exceed the buffer's {self.max_pairs}")
        if n:
            self.field("src_dst_pairs", n).copy_(torch.as_tensor(pairs, dtype=torch.int32).reshape(n, 2))
        self.num_pairs = n
        return nat.step_layout(self.num_seqs, self.eng.num_q_heads, self.eng.num_kv_heads, self.eng.head_dim,
                               self.width, n)["bytes"]

    def h2d_bytes(self) -> int:
        """Bytes the staging kernel brings across the host link for the packed
        step: every field but the block tables whole, and of each table row
        the 16-byte words holding its entries up to ceil(context_len / 16)."""
        lay = nat.step_layout(self.num_seqs, self.eng.num_q_heads, self.eng.num_kv_heads, self.eng.head_dim,
                              self.width, self.num_pairs)
        dense = lay["bytes"] - (lay["context_lens"] - lay["block_tables"])
        ctx = self.field("context_lens").numpy().astype(np.int64)
        live = np.minimum(np.maximum((ctx + nat.BLOCK_TOKENS - 1) // nat.BLOCK_TOKENS, 0), self.width)
        start = lay["block_tables"] + np.arange(self.num_seqs, dtype=np.int64) * self.width * 4
        words = np.where(live > 0, (start + live * 4 + 15) // 16 - start // 16, 0)
        return int(dense + 16 * words.sum())

    def run(self, scale: float, num_ctas: int = 0, stream=None) -> torch.Tensor:
        """Enqueue the step; out_host holds the output once the stream passes it."""
        e = self.eng
        nat.decode_step_host(self.host, self.staging, self.num_pairs, e.k_cache, e.v_cache, self.width,
                             self.num_seqs, e.num_q_heads, scale, self.workspace, self.out_dev, self.out_host,
                             e.error, num_ctas, stream)
        return self.out_host
