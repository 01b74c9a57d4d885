"""Block manager policy, restated as plain Python.

Sources:
  - cs2680 Lecture 10, §10.3: a pool of fixed-size blocks, a block table per
    sequence, growth by one table entry; §10.4: blocks shared by reference
    count, copied only on divergence (refcount 8 -> 7 + 1 when one branch
    writes).
  - "KV cache systems", copy-on-write paragraph: the first request to write a
    shared block triggers the copy; only the divergent suffix takes memory.
  - "Reserve the page a request has not written yet": reserve
    ceil((prompt + max_output) / 16) pages at admission ("Separate the pool
    from its owners"); reserve-and-admit is one serialised decision ("Pick a
    reservation policy you can explain"); shared complete prefix pages are
    charged once, each private suffix still needs its own pages ("Charge
    shared pages once"); freeing changes ownership, not device memory.

Readings where the pages are silent (each is a policy choice both
implementations share):
  - free list: a stack; blocks are handed out in `free_order` (ascending ids
    by default) and a released block is the next one handed out;
  - a prefix group shares only the complete pages of its prefix
    (prefix_len // 16); a partial prefix page is private to each member;
  - fork shares the parent's written blocks; if the parent's last written
    block is partial, each child reserves one spare page for the copy that
    its (or a sibling's) first write will need, so that a shared partial
    block b always holds refcount(b) - 1 spares and copy-on-write never fails;
  - copy-on-write: the writer takes a spare and becomes the block's new
    owner; a writer that sees refcount 1 writes in place;
  - a call that fails changes no state.
"""
from __future__ import annotations


class BlockManagerError(Exception):
    pass


class InvalidRequest(BlockManagerError):
    pass


class PoolExhausted(BlockManagerError):
    """Admission or fork refused: too few free pages."""


class ReservationExceeded(BlockManagerError):
    """An append past the pages the sequence reserved."""


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


class _Seq:
    __slots__ = ("table", "ctx", "group")

    def __init__(self, table, ctx, group):
        self.table, self.ctx, self.group = table, ctx, group


class BlockManager:
    def __init__(self, num_blocks: int, block_tokens: int = 16, free_order=None):
        if num_blocks <= 0 or block_tokens <= 0:
            raise InvalidRequest("num_blocks and block_tokens must be positive")
        order = list(range(num_blocks)) if free_order is None else [int(x) for x in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise InvalidRequest("free_order must be a permutation of the pool")
        self.num_blocks = num_blocks
        self.b = block_tokens
        self._free = order[::-1]  # pop() yields order[0] first
        self.ref = [0] * num_blocks
        self.spares: dict[int, list[int]] = {}
        self.seqs: dict[int, _Seq] = {}
        self.groups: dict[int, dict] = {}
        self.next_id = 0
        self.cow_copies = 0

    # -- helpers ---------------------------------------------------------
    def _pop(self) -> int:
        return self._free.pop()

    def _push(self, blk: int) -> None:
        self._free.append(blk)

    @property
    def num_free(self) -> int:
        return len(self._free)

    # -- admission -------------------------------------------------------
    def admit(self, prompt_len: int, max_new: int, group: int = -1, prefix_len: int = 0) -> int:
        """Reserve every page the request can ever fill and admit it, or refuse."""
        if prompt_len < 0 or max_new < 0 or prompt_len + max_new <= 0:
            raise InvalidRequest("need prompt_len >= 0, max_new >= 0, and at least one token")
        total = _ceil_div(prompt_len + max_new, self.b)
        n_shared, shared = 0, []
        if group >= 0:
            if prefix_len < 0 or prefix_len > prompt_len:
                raise InvalidRequest("prefix_len must lie within the prompt")
            n_shared = prefix_len // self.b
            g = self.groups.get(group)
            if g is not None:
                if g["prefix_len"] != prefix_len:
                    raise InvalidRequest("a prefix group has one prefix length")
                shared = g["pages"]
        need = total - len(shared)
        if need > self.num_free:
            raise PoolExhausted(f"need {need} pages, {self.num_free} free")
        if group >= 0 and group not in self.groups:
            shared = [self._pop() for _ in range(n_shared)]
            self.groups[group] = {"pages": shared, "prefix_len": prefix_len, "members": 0}
        table = list(shared) + [self._pop() for _ in range(total - len(shared))]
        for blk in table:
            self.ref[blk] += 1
        if group >= 0:
            self.groups[group]["members"] += 1
        sid = self.next_id
        self.next_id += 1
        self.seqs[sid] = _Seq(table, prompt_len, group)
        return sid

    def fork(self, parent: int, n: int) -> list[int]:
        """n children share the parent's written blocks; each reserves its own
        pages for the rest of the allowance (plus a spare for a partial block)."""
        if parent not in self.seqs or n < 0:
            raise InvalidRequest("unknown parent or negative n")
        p = self.seqs[parent]
        written = _ceil_div(p.ctx, self.b)
        partial = p.ctx % self.b != 0
        per_child = (len(p.table) - written) + (1 if partial else 0)
        if n * per_child > self.num_free:
            raise PoolExhausted(f"need {n * per_child} pages, {self.num_free} free")
        kids = []
        for _ in range(n):
            table = p.table[:written] + [self._pop() for _ in range(len(p.table) - written)]
            for blk in table:
                self.ref[blk] += 1
            if partial:
                self.spares.setdefault(p.table[written - 1], []).append(self._pop())
            if p.group >= 0:
                self.groups[p.group]["members"] += 1
            sid = self.next_id
            self.next_id += 1
            self.seqs[sid] = _Seq(table, p.ctx, p.group)
            kids.append(sid)
        return kids

    # -- decode-step bookkeeping ------------------------------------------
    def prepare_append(self, seq_ids):
        """Slot for each sequence's next token, and the (src, dst) block copies
        that must run before the tokens are written. Sequences are handled in
        the given order."""
        seq_ids = [int(s) for s in seq_ids]
        if len(set(seq_ids)) != len(seq_ids) or any(s not in self.seqs for s in seq_ids):
            raise InvalidRequest("unknown or repeated sequence id")
        for sid in seq_ids:
            s = self.seqs[sid]
            if s.ctx // self.b >= len(s.table):
                raise ReservationExceeded(f"sequence {sid} is at its reserved length")
        slots, pairs = [], []
        for sid in seq_ids:
            s = self.seqs[sid]
            lb = s.ctx // self.b
            blk = s.table[lb]
            if self.ref[blk] > 1:
                spare = self.spares.get(blk)
                if not spare:
                    raise BlockManagerError("shared block without a reserved spare")
                dst = spare.pop()
                if not spare:
                    del self.spares[blk]
                self.ref[blk] -= 1
                self.ref[dst] = 1
                s.table[lb] = dst
                pairs.append((blk, dst))
                self.cow_copies += 1
                blk = dst
            slots.append(blk * self.b + s.ctx % self.b)
            s.ctx += 1
        return slots, pairs

    def free(self, sid: int) -> None:
        """Release a sequence's references; blocks that reach refcount 0 (and
        spares no longer needed) go back to the free list."""
        if sid not in self.seqs:
            raise InvalidRequest("unknown sequence")
        s = self.seqs.pop(sid)
        for blk in s.table:
            self.ref[blk] -= 1
            sp = self.spares.get(blk)
            if sp and len(sp) > self.ref[blk] - 1:
                self._push(sp.pop())
                if not sp:
                    del self.spares[blk]
            if self.ref[blk] == 0:
                self._push(blk)
        if s.group >= 0:
            g = self.groups[s.group]
            g["members"] -= 1
            if g["members"] == 0:
                del self.groups[s.group]

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
        }
