"""Pins for the oracle's accounting and block manager: the pages' worked
numbers (tests/golden/worked_numbers.json) and brute-force invariants."""
import random

import pytest

from oracle import accounting as acc
from oracle.block_manager import (BlockManager, InvalidRequest, PoolExhausted,
                                  ReservationExceeded)


def test_admission_arithmetic(golden):
    g = golden["admission_32L"]
    kv = acc.kv_bytes_per_token(g["n_layers"], g["n_kv_heads"], g["head_dim"], g["bytes_per_elem"])
    assert kv == g["kv_bytes_per_token"]
    page = acc.page_bytes(g["tokens_per_page"], kv)
    assert page == g["page_bytes"]
    assert acc.pool_pages(g["pool_bytes"], page) == g["pool_pages"]
    pages = acc.request_pages(g["prompt_tokens"], g["output_tokens"])
    assert pages == g["request_pages"] and pages not in g["wrong_answers"]
    assert acc.request_pages(g["prompt_tokens"], 0) == g["prompt_only_pages"]
    assert acc.group_pages(8, g["prompt_tokens"], g["output_tokens"]) == g["eight_shared_pages"]
    assert 8 * pages == g["eight_unshared_pages"]
    assert acc.group_pages(7, g["prompt_tokens"], g["output_tokens"]) == g["seven_shared_pages"]
    shared = g["shared_prefix_pages"]
    private = g["private_pages_per_request"]
    assert acc.max_admitted(g["pool_pages"], shared + private, private) == g["admitted_shared"]
    assert acc.max_admitted(g["pool_pages"], pages, pages) == g["admitted_isolated"]


def test_kv_bytes_70b(golden):
    g = golden["kv_70b"]
    assert acc.kv_bytes_per_token(g["n_layers"], g["n_kv_heads"], g["head_dim"], g["bytes_per_elem"]) == g["kv_bytes_per_token"]


def test_block_manager_shared_prefix_admission(golden):
    g = golden["admission_32L"]
    bm = BlockManager(g["pool_pages"])
    ids = [bm.admit(g["prompt_tokens"], g["output_tokens"], 0, g["prompt_tokens"]) for _ in range(g["admitted_shared"])]
    assert len(ids) == 7
    st = bm.stats()
    assert st["used"] == g["seven_shared_pages"] and st["free"] == g["seven_shared_free_after"]
    assert st["shared"] == g["shared_prefix_pages"]
    assert all(bm.ref[b] == 7 for b in bm.table(ids[0])[: g["shared_prefix_pages"]])
    with pytest.raises(PoolExhausted):
        bm.admit(g["prompt_tokens"], g["output_tokens"], 0, g["prompt_tokens"])
    assert bm.stats() == st  # a refused admission changes nothing


def test_block_manager_isolated_admission(golden):
    g = golden["admission_32L"]
    bm = BlockManager(g["pool_pages"])
    bm.admit(g["prompt_tokens"], g["output_tokens"], 0, g["prompt_tokens"])
    assert bm.stats()["used"] == g["request_pages"]
    with pytest.raises(PoolExhausted):
        bm.admit(g["prompt_tokens"], g["output_tokens"], 1, g["prompt_tokens"])
    with pytest.raises(PoolExhausted):
        bm.admit(g["prompt_tokens"], g["output_tokens"])
    assert bm.stats()["free"] == g["pool_pages"] - g["request_pages"]


def test_fanout_sharing_n8(golden):
    g = golden["fanout_n8"]
    bm = BlockManager(4096)
    parent = bm.admit(g["prompt_tokens"], g["output_tokens"])
    bm.fork(parent, g["samples"] - 1)
    assert bm.stats()["used"] * 16 == g["shared_tokens"]
    solo = BlockManager(4096)
    for _ in range(g["samples"]):
        solo.admit(g["prompt_tokens"], g["output_tokens"])
    assert solo.stats()["used"] * 16 == g["unshared_tokens"]
    assert round(g["unshared_tokens"] / g["shared_tokens"], 1) == g["ratio_rounded"]


def test_fanout_sharing_n16_bytes(golden):
    g = golden["fanout_n16"]
    bm = BlockManager(16384)
    parent = bm.admit(g["prompt_tokens"], g["output_tokens"])
    bm.fork(parent, g["samples"] - 1)
    shared = bm.stats()["used"] * 16 * g["kv_bytes_per_token"]
    unshared = g["samples"] * acc.request_pages(g["prompt_tokens"], g["output_tokens"]) * 16 * g["kv_bytes_per_token"]
    assert round(unshared / 1e9, 1) == g["unshared_gb_rounded"]
    assert round(shared / 1e9, 1) == g["shared_gb_rounded"]
    assert round(unshared / shared, 1) == g["ratio_rounded"]


def test_tail_waste(golden):
    g = golden["tail_waste"]
    b = g["block_tokens"]
    wastes = [acc.tail_waste(d, b) for d in range(1, 16 * b + 1)]
    assert min(wastes) == 0 and max(wastes) == g["max_waste"]
    assert sum(wastes) / len(wastes) == g["mean_waste_uniform"]


def test_table_entries(golden):
    g = golden["table_entries"]
    assert acc.table_entries(8192) == g["entries_8k_b16"]
    assert acc.table_entries(8192) * 4 == g["bytes_8k_b16"]
    assert acc.table_entries(8192, 64) == g["entries_8k_b64"]
    assert acc.table_entries(4096) == g["entries_4k_b16"]


def test_copy_on_write_refcount_board():
    # cs2680 §10.4: eight branches share a block (refcount 8); one branch
    # writes a token and gets its own block (refcount 7 + 1).
    bm = BlockManager(64)
    parent = bm.admit(20, 12)  # ctx 20: block 1 is partial
    kids = bm.fork(parent, 7)
    shared = bm.table(parent)[1]
    assert bm.ref[shared] == 8
    slots, pairs = bm.prepare_append([kids[3]])
    (src, dst), = pairs
    assert src == shared and bm.ref[shared] == 7 and bm.ref[dst] == 1
    assert slots == [dst * 16 + 4]
    assert bm.table(kids[3])[1] == dst
    # the remaining sharers copy in turn; the last writes in place
    slots, pairs = bm.prepare_append([parent] + [k for k in kids if k != kids[3]])
    assert len(pairs) == 6 and bm.ref[shared] == 1
    assert slots[-1] == shared * 16 + 4
    assert bm.stats()["spares"] == 0 and bm.stats()["cow_copies"] == 7


def test_full_blocks_are_never_copied():
    bm = BlockManager(64)
    parent = bm.admit(32, 16)  # two full prompt blocks
    kids = bm.fork(parent, 3)
    slots, pairs = bm.prepare_append([parent] + kids)
    assert pairs == [] and len(set(s // 16 for s in slots)) == 4


def test_reservation_limit():
    bm = BlockManager(8)
    s = bm.admit(15, 1)
    bm.prepare_append([s])
    with pytest.raises(ReservationExceeded):
        bm.prepare_append([s])


def test_invalid_calls_change_nothing():
    bm = BlockManager(8)
    s = bm.admit(3, 3)
    st = bm.stats()
    for call in (lambda: bm.admit(-1, 3), lambda: bm.admit(0, 0), lambda: bm.fork(99, 1),
                 lambda: bm.prepare_append([s, s]), lambda: bm.admit(3, 3, 0, 4)):
        with pytest.raises(InvalidRequest):
            call()
    assert bm.stats() == st


def test_free_returns_pages_lifo():
    bm = BlockManager(10)
    a = bm.admit(30, 2)  # blocks 0, 1
    bm.admit(16, 0)  # block 2
    bm.free(a)
    assert bm.stats()["free"] == 9
    c = bm.admit(1, 0)
    assert bm.table(c) == [1]  # last released, first reused


def _check_invariants(bm):
    st = bm.stats()
    referenced = {b for s in bm.seqs.values() for b in s.table}
    spare = {b for v in bm.spares.values() for b in v}
    free = set(bm._free)
    assert len(free) == len(bm._free)
    assert not (free & referenced) and not (free & spare) and not (spare & referenced)
    assert st["free"] + st["used"] + st["spares"] == bm.num_blocks
    assert st["ref_sum"] == sum(len(s.table) for s in bm.seqs.values())
    for b, v in bm.spares.items():
        assert len(v) == bm.ref[b] - 1


def test_random_operations_keep_invariants():
    rnd = random.Random(0)
    for trial in range(20):
        n = rnd.randint(20, 200)
        bm = BlockManager(n, free_order=rnd.sample(range(n), n) if trial % 2 else None)
        for _ in range(300):
            op = rnd.random()
            try:
                if op < 0.3 or not bm.seqs:
                    grp = rnd.choice([-1, -1, 0, 1])
                    p = rnd.randint(0, 60)
                    bm.admit(p, rnd.randint(1, 40), grp, 32 if grp >= 0 and p >= 32 else 0)
                elif op < 0.45:
                    bm.fork(rnd.choice(list(bm.seqs)), rnd.randint(1, 3))
                elif op < 0.85:
                    ids = rnd.sample(list(bm.seqs), rnd.randint(1, len(bm.seqs)))
                    bm.prepare_append(ids)
                else:
                    bm.free(rnd.choice(list(bm.seqs)))
            except (PoolExhausted, ReservationExceeded, InvalidRequest):
                pass
            _check_invariants(bm)
        for s in list(bm.seqs):
            bm.free(s)
        assert bm.stats()["free"] == bm.num_blocks and not bm.groups
