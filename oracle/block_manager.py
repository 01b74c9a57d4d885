"""Block manager policy, restated as plain Python.

Sources:
  - cs2680 Lecture 10, §10.3: a pool of fixed-size blocks, a block table per
    sequence, growth by one table entry; §10.4: blocks shared by reference
    count, copied only on divergence (refcount 8 -> 7 + 1 when one branch
    writes); §10.5: blocks handed out on demand can run out, and the engine
    then refuses new arrivals or preempts a resident sequence, keeping a
    watermark of free blocks so that preemption is rare; a preempted
    sequence loses its cache, not its tokens, and is recomputed.
  - "KV cache systems", copy-on-write paragraph: the first request to write a
    shared block triggers the copy; only the divergent suffix takes memory.
    Prefix-hit paragraph: a block of b tokens is reusable iff all b tokens
    match and all preceding blocks matched (8,000 matching tokens reuse
    floor(8000 / 16) = 500 blocks). Eviction paragraph: blocks pinned by
    in-flight requests are never evicted, and a cached block is evicted only
    when no cached block extends it (leaf first).
  - "Reserve the page a request has not written yet": reserve
    ceil((prompt + max_output) / 16) pages at admission ("Separate the pool
    from its owners"); an incremental policy admits more requests and must
    say what happens when no page is available ("Pick a reservation policy
    you can explain"); reserve-and-admit is one serialised decision; shared
    complete prefix pages are charged once, each private suffix still needs
    its own pages ("Charge shared pages once"); freeing changes ownership,
    not device memory.

Readings where the pages are silent (each is a policy choice both
implementations share):
  - free list: a stack; blocks are handed out in `free_order` (ascending ids
    by default) and a released block is the next one handed out;
  - a prefix group shares only the complete pages of its prefix
    (prefix_len // b); a partial prefix page is private to each member;
  - full reservation (default): admission reserves every page the request
    can fill; fork shares the parent's written blocks and each child reserves
    the rest of its allowance plus, when the parent's last written block is
    partial, one spare page for the copy its (or a sibling's) first write
    will need, so that a shared partial block b always holds refcount(b) - 1
    spares and copy-on-write never fails;
  - incremental: admission reserves the prompt's pages only and must leave
    `watermark` pages available; a token that starts a new block, or a write
    into a shared block, takes a page then; a step whose pages are not all
    available fails as a whole (no state change) and the caller preempts;
  - copy-on-write: the writer takes a spare (or a new page) and becomes the
    block's new owner; a writer that sees refcount 1 writes in place;
  - preemption releases the sequence's blocks and keeps its token count;
    resuming reserves fresh private pages (as admission would, watermark
    included) for the caller to recompute; the preemption victim offered is
    the newest running sequence;
  - prefix cache: every complete prompt block of a request admitted with its
    tokens is indexed by its exact token prefix; a released indexed block is
    kept (not freed) until evicted; allocation takes free blocks first, then
    evicts the least recently released indexed block that no indexed block
    extends; pages held by the cache count as available;
  - a call that fails changes no state.
"""
from __future__ import annotations


class BlockManagerError(Exception):
    pass


class InvalidRequest(BlockManagerError):
    pass


class PoolExhausted(BlockManagerError):
    """Admission, fork, growth or resume refused: too few available pages."""


class ReservationExceeded(BlockManagerError):
    """An append past the pages the sequence reserved (full reservation)."""


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


class _Seq:
    __slots__ = ("table", "ctx", "group", "max_len", "running")

    def __init__(self, table, ctx, group, max_len):
        self.table, self.ctx, self.group, self.max_len = table, ctx, group, max_len
        self.running = True


class BlockManager:
    def __init__(self, num_blocks: int, block_tokens: int = 16, free_order=None, incremental: bool = False,
                 watermark: int = 0, prefix_cache: bool = False):
        if num_blocks <= 0 or block_tokens <= 0 or watermark < 0:
            raise InvalidRequest("num_blocks and block_tokens must be positive, watermark >= 0")
        order = list(range(num_blocks)) if free_order is None else [int(x) for x in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise InvalidRequest("free_order must be a permutation of the pool")
        self.num_blocks = num_blocks
        self.b = block_tokens
        self.incremental, self.watermark, self.prefix_cache = bool(incremental), int(watermark), bool(prefix_cache)
        self._free = order[::-1]  # pop() yields order[0] first
        self.ref = [0] * num_blocks
        self.spares: dict[int, list[int]] = {}
        self.seqs: dict[int, _Seq] = {}
        self.groups: dict[int, dict] = {}
        self.next_id = 0
        self.cow_copies = 0
        # prefix cache: exact token prefix -> block, and per indexed block its
        # key, parent block, number of indexed children and release time
        self.index: dict[tuple, int] = {}
        self.key: dict[int, tuple] = {}
        self.parent: dict[int, int] = {}
        self.children: dict[int, int] = {}
        self.last_use: dict[int, int] = {}
        self.clock = 0
        self.cache_hits = 0
        self.evictions = 0
        self.reused: dict[int, int] = {}

    # -- pages -----------------------------------------------------------
    @property
    def num_free(self) -> int:
        return len(self._free)

    def _cached_idle(self) -> int:
        return sum(1 for blk in self.key if self.ref[blk] == 0)

    def available(self) -> int:
        """Pages that can be handed out: free ones and idle cached ones."""
        return len(self._free) + self._cached_idle()

    def _victim(self) -> int:
        """The idle cached block no cached block extends, least recently released."""
        leaves = [blk for blk in self.key if self.ref[blk] == 0 and self.children.get(blk, 0) == 0]
        if not leaves:
            raise BlockManagerError("no page available")
        return min(leaves, key=lambda blk: (self.last_use[blk], blk))

    def _alloc(self) -> int:
        if self._free:
            return self._free.pop()
        victim = self._victim()
        del self.index[self.key.pop(victim)]
        par = self.parent.pop(victim)
        if par >= 0:
            self.children[par] -= 1
        self.children.pop(victim, None)
        self.last_use.pop(victim, None)
        self.evictions += 1
        return victim

    def _release(self, table) -> None:
        for blk in table:
            self.ref[blk] -= 1
            sp = self.spares.get(blk)
            if sp and len(sp) > self.ref[blk] - 1:
                self._free.append(sp.pop())
                if not sp:
                    del self.spares[blk]
            if self.ref[blk] == 0:
                if blk in self.key:
                    self.clock += 1
                    self.last_use[blk] = self.clock
                else:
                    self._free.append(blk)

    # -- prefix index ------------------------------------------------------
    def _block_key(self, tokens, i: int) -> tuple:
        """Block i of a prompt is identified by every token up to its end."""
        return tuple(tokens[: self.b * (i + 1)])

    def _lookup(self, tokens) -> list[int]:
        """Cached blocks for the prompt's complete blocks, from the first up to
        the first miss."""
        hits = []
        for i in range(len(tokens) // self.b):
            blk = self.index.get(self._block_key(tokens, i))
            if blk is None:
                break
            hits.append(blk)
        return hits

    def _room(self, hits) -> int:
        """Pages an admission can take: the available ones, less the idle
        cached blocks it is about to reuse."""
        return self.available() - sum(1 for blk in hits if self.ref[blk] == 0)

    # -- admission -------------------------------------------------------
    def admit(self, prompt_len: int, max_new: int, group: int = -1, prefix_len: int = 0, tokens=None) -> int:
        """Reserve the pages the policy charges and admit the request, or refuse."""
        if prompt_len < 0 or max_new < 0 or prompt_len + max_new <= 0:
            raise InvalidRequest("need prompt_len >= 0, max_new >= 0, and at least one token")
        if tokens is not None:
            tokens = [int(t) for t in tokens]
            if not self.prefix_cache or group >= 0 or len(tokens) != prompt_len:
                raise InvalidRequest("tokens need the prefix cache, no group, and one token per prompt position")
        total = _ceil_div(prompt_len if self.incremental else prompt_len + max_new, self.b)
        shared, hits, new_group = [], [], False
        if group >= 0:
            if prefix_len < 0 or prefix_len > prompt_len:
                raise InvalidRequest("prefix_len must lie within the prompt")
            g = self.groups.get(group)
            if g is not None:
                if g["prefix_len"] != prefix_len:
                    raise InvalidRequest("a prefix group has one prefix length")
                shared = list(g["pages"])
            else:
                new_group = True
        if tokens is not None:
            hits = self._lookup(tokens)
            shared = hits
        need = total - len(shared)
        if need + self.watermark > self._room(hits):
            raise PoolExhausted(f"need {need} pages (+{self.watermark} watermark), {self._room(hits)} available")
        if new_group:
            shared = [self._alloc() for _ in range(prefix_len // self.b)]
            self.groups[group] = {"pages": list(shared), "prefix_len": prefix_len, "members": 0}
        for blk in hits:
            self.ref[blk] += 1  # an idle cached block is in use again
        table = list(shared) + [self._alloc() for _ in range(total - len(shared))]
        for blk in table[len(hits):]:
            self.ref[blk] += 1
        if group >= 0:
            self.groups[group]["members"] += 1
        if tokens is not None:
            for i in range(len(hits), prompt_len // self.b):
                blk = table[i]
                k = self._block_key(tokens, i)
                self.index[k] = blk
                self.key[blk] = k
                self.parent[blk] = table[i - 1] if i > 0 else -1
                self.children.setdefault(blk, 0)
                if i > 0:
                    self.children[table[i - 1]] = self.children.get(table[i - 1], 0) + 1
            self.cache_hits += len(hits)
        sid = self.next_id
        self.next_id += 1
        self.seqs[sid] = _Seq(table, prompt_len, group, prompt_len + max_new)
        self.reused[sid] = len(hits)
        return sid

    def fork(self, parent: int, n: int) -> list[int]:
        """n children share the parent's written blocks; under full reservation
        each reserves its own pages for the rest of the allowance (plus a spare
        for a partial block)."""
        if parent not in self.seqs or not self.seqs[parent].running or n < 0:
            raise InvalidRequest("unknown or preempted parent, or negative n")
        p = self.seqs[parent]
        written = _ceil_div(p.ctx, self.b)
        partial = p.ctx % self.b != 0 and not self.incremental
        per_child = 0 if self.incremental else (len(p.table) - written) + (1 if partial else 0)
        if n * per_child > self.available():
            raise PoolExhausted(f"need {n * per_child} pages, {self.available()} available")
        kids = []
        for _ in range(n):
            table = p.table[:written] + [self._alloc() for _ in range(len(p.table) - written)]
            for blk in table:
                self.ref[blk] += 1
            if partial:
                self.spares.setdefault(p.table[written - 1], []).append(self._alloc())
            if p.group >= 0:
                self.groups[p.group]["members"] += 1
            sid = self.next_id
            self.next_id += 1
            self.seqs[sid] = _Seq(table, p.ctx, p.group, p.max_len)
            self.reused[sid] = 0
            kids.append(sid)
        return kids

    # -- decode-step bookkeeping ------------------------------------------
    def prepare_append(self, seq_ids):
        """Slot for each sequence's next token, and the (src, dst) block copies
        that must run before the tokens are written. Sequences are handled in
        the given order."""
        seq_ids = [int(s) for s in seq_ids]
        if len(set(seq_ids)) != len(seq_ids) or any(s not in self.seqs or not self.seqs[s].running
                                                    for s in seq_ids):
            raise InvalidRequest("unknown, preempted or repeated sequence id")
        need, ref_left, spare_left = 0, {}, {}
        for sid in seq_ids:
            s = self.seqs[sid]
            lb = s.ctx // self.b
            if lb >= len(s.table):
                if not self.incremental:
                    raise ReservationExceeded(f"sequence {sid} is at its reserved length")
                need += 1
                continue
            blk = s.table[lb]
            r = ref_left.setdefault(blk, self.ref[blk])
            sp = spare_left.setdefault(blk, len(self.spares.get(blk, [])))
            if r > 1:
                ref_left[blk] = r - 1
                if sp > 0:
                    spare_left[blk] = sp - 1
                elif self.incremental:
                    need += 1
                else:
                    raise BlockManagerError("shared block without a reserved spare")
        if need > self.available():
            raise PoolExhausted(f"the step needs {need} pages, {self.available()} available")
        slots, pairs = [], []
        for sid in seq_ids:
            s = self.seqs[sid]
            lb = s.ctx // self.b
            if lb >= len(s.table):
                blk = self._alloc()
                self.ref[blk] = 1
                s.table.append(blk)
            blk = s.table[lb]
            if self.ref[blk] > 1:
                spare = self.spares.get(blk)
                if spare:
                    dst = spare.pop()
                    if not spare:
                        del self.spares[blk]
                else:
                    dst = self._alloc()
                self.ref[blk] -= 1
                self.ref[dst] = 1
                s.table[lb] = dst
                pairs.append((blk, dst))
                self.cow_copies += 1
                blk = dst
            slots.append(blk * self.b + s.ctx % self.b)
            s.ctx += 1
        return slots, pairs

    def _leave_group(self, s: _Seq) -> None:
        if s.group >= 0:
            g = self.groups[s.group]
            g["members"] -= 1
            if g["members"] == 0:
                del self.groups[s.group]
            s.group = -1

    def free(self, sid: int) -> None:
        """Release a sequence's references; blocks that reach refcount 0 go
        back to the free list (or stay cached), spares no longer needed too."""
        if sid not in self.seqs:
            raise InvalidRequest("unknown sequence")
        s = self.seqs.pop(sid)
        self.reused.pop(sid, None)
        if s.running:
            self._release(s.table)
            self._leave_group(s)

    def preempt(self, sid: int) -> int:
        """Release a running sequence's blocks, keeping its token count;
        returns the number of its table entries released."""
        if sid not in self.seqs or not self.seqs[sid].running:
            raise InvalidRequest("unknown or already preempted sequence")
        s = self.seqs[sid]
        n = len(s.table)
        self._release(s.table)
        self._leave_group(s)
        s.table = []
        s.running = False
        return n

    def resume(self, sid: int) -> None:
        """Re-admit a preempted sequence on fresh private pages, for the caller
        to recompute its KV."""
        if sid not in self.seqs or self.seqs[sid].running:
            raise InvalidRequest("unknown or running sequence")
        s = self.seqs[sid]
        total = _ceil_div(s.ctx if self.incremental else s.max_len, self.b)
        if total + self.watermark > self.available():
            raise PoolExhausted(f"need {total} pages (+{self.watermark} watermark), {self.available()} available")
        s.table = [self._alloc() for _ in range(total)]
        for blk in s.table:
            self.ref[blk] = 1
        s.running = True

    def slots(self, sid: int, first: int, n: int) -> list[int]:
        """Slots of a running sequence's token positions [first, first + n),
        within its table: where a prefill or a recompute writes their KV."""
        s = self.seqs.get(sid)
        if s is None or not s.running or first < 0 or n < 0 or first + n > len(s.table) * self.b:
            raise InvalidRequest("unknown or preempted sequence, or positions outside its table")
        return [s.table[p // self.b] * self.b + p % self.b for p in range(first, first + n)]

    def newest_running(self) -> int:
        running = [sid for sid, s in self.seqs.items() if s.running]
        return max(running) if running else -1

    # -- queries -----------------------------------------------------------
    def table(self, sid: int) -> list[int]:
        return list(self.seqs[sid].table)

    def context_len(self, sid: int) -> int:
        return self.seqs[sid].ctx

    def stats(self) -> dict:
        return {
            "free": self.num_free,
            "used": sum(1 for r in self.ref if r > 0),
            "shared": sum(1 for r in self.ref if r > 1),
            "ref_sum": sum(self.ref),
            "spares": sum(len(v) for v in self.spares.values()),
            "cow_copies": self.cow_copies,
            "seqs": len(self.seqs),
            "cached": len(self.key),
            "cached_idle": self._cached_idle(),
            "available": self.available(),
            "cache_hits": self.cache_hits,
            "evictions": self.evictions,
            "preempted": sum(1 for s in self.seqs.values() if not s.running),
        }
