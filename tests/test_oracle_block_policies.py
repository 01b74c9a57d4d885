"""Pins for the oracle block manager's incremental policy (watermark,
preemption by recompute) and its prefix-cache index: the pages' worked
numbers, closed forms derived from them, brute force over tiny vocabularies
and structural invariants. CPU only."""
import random

import pytest

from oracle.block_manager import BlockManager, InvalidRequest, PoolExhausted


def _lcp(a, b):
    n = 0
    for x, y in zip(a, b):
        if x != y:
            break
        n += 1
    return n


def _check_invariants(bm: BlockManager):
    st = bm.stats()
    # every page is exactly one of: free, referenced, a reserved spare, idle in the cache
    assert st["free"] + st["used"] + st["spares"] + st["cached_idle"] == bm.num_blocks
    assert st["ref_sum"] == sum(len(s.table) for s in bm.seqs.values() if s.running)
    assert all(not s.table for s in bm.seqs.values() if not s.running)
    assert st["available"] == st["free"] + st["cached_idle"]
    free = set(bm._free)
    assert len(free) == len(bm._free)
    for blk in range(bm.num_blocks):
        if blk in free:
            assert bm.ref[blk] == 0 and blk not in bm.key
    # the index is prefix-closed and its child counts are exact
    kids = {}
    for blk, k in bm.key.items():
        assert bm.index[k] == blk and len(k) % bm.b == 0
        par = bm.parent[blk]
        if len(k) == bm.b:
            assert par == -1
        else:
            assert bm.key[par] == k[:-bm.b]
            kids[par] = kids.get(par, 0) + 1
            if bm.ref[blk] > 0:
                assert bm.ref[par] > 0  # a block in use pins its ancestors
    for blk in bm.key:
        assert bm.children.get(blk, 0) == kids.get(blk, 0)


# -- prefix cache ----------------------------------------------------------

def test_prefix_hit_worked_example(golden):
    g = golden["prefix_hit_8000"]
    b, m = g["block_tokens"], g["matching_tokens"]
    rnd = random.Random(0)
    cached = [rnd.randrange(32000) for _ in range(m + 200)]
    bm = BlockManager(2048, b, prefix_cache=True)
    bm.admit(len(cached), 1, tokens=cached)
    for differ_at, expect in [(m, g["reused_blocks"]), (m + b - 1, g["reused_blocks"]),
                              (m - 1, g["reused_blocks"] - 1)]:
        req = list(cached)
        req[differ_at] = (req[differ_at] + 1) % 32000
        sid = bm.admit(len(req), 1, tokens=req)
        assert bm.reused[sid] == expect
        assert bm.table(sid)[:expect] == bm.table(0)[:expect]
        bm.free(sid)
        _check_invariants(bm)


def test_two_users_share_system_prompt(golden):
    g = golden["shared_system_prompt_2000"]
    b = g["block_tokens"]
    rnd = random.Random(1)
    system = [rnd.randrange(32000) for _ in range(g["system_prompt_tokens"])]
    bm = BlockManager(1024, b, prefix_cache=True)
    a = bm.admit(len(system) + 300, 64, tokens=system + [1] * 300)
    c = bm.admit(len(system) + 100, 64, tokens=system + [2] * 100)
    assert bm.reused[c] == g["shared_blocks"]
    assert bm.stats()["shared"] == g["shared_blocks"]
    assert all(bm.ref[blk] == 2 for blk in bm.table(a)[: g["shared_blocks"]])
    # block 125 holds tokens 2000..2015: the users' texts differ there
    assert bm.table(a)[g["shared_blocks"]] != bm.table(c)[g["shared_blocks"]]


def test_hits_are_prefix_only():
    bm = BlockManager(256, 16, prefix_cache=True)
    base = list(range(160))  # 10 complete blocks
    bm.admit(len(base), 0, tokens=base)
    bad = list(base)
    bad[5 * 16 + 3] = -1  # block 5 differs, blocks 6..9 match again
    sid = bm.admit(len(bad), 0, tokens=bad)
    assert bm.reused[sid] == 5
    first = list(base)
    first[0] = -1
    assert bm.reused[bm.admit(len(first), 0, tokens=first)] == 0
    _check_invariants(bm)


def test_partial_prompt_block_is_not_indexed():
    bm = BlockManager(64, 16, prefix_cache=True)
    p = list(range(40))
    a = bm.admit(40, 8, tokens=p)
    assert bm.stats()["cached"] == 2
    c = bm.admit(40, 8, tokens=p)
    assert bm.reused[c] == 2
    assert bm.table(c)[:2] == bm.table(a)[:2] and bm.table(c)[2] != bm.table(a)[2]
    # the shared full blocks are never written: the next token lands in block 2
    slots, pairs = bm.prepare_append([a, c])
    assert pairs == [] and [s // 16 for s in slots] == [bm.table(a)[2], bm.table(c)[2]]


@pytest.mark.parametrize("seed", range(6))
def test_hits_match_brute_force(seed):
    """Without eviction, a prompt reuses max over earlier prompts of
    floor(common prefix / b) blocks, and the index holds one block per
    distinct complete-block prefix."""
    rnd = random.Random(seed)
    b = 4
    bm = BlockManager(4096, b, prefix_cache=True)
    seen, live = [], []
    for _ in range(80):
        if live and rnd.random() < 0.3:
            bm.free(live.pop(rnd.randrange(len(live))))  # cached blocks outlive their owner
        n = rnd.randint(1, 30)
        if seen and rnd.random() < 0.7:
            src = rnd.choice(seen)
            keep = rnd.randint(0, len(src))
            p = src[:keep] + [rnd.randrange(2) for _ in range(max(0, n - keep))]
        else:
            p = [rnd.randrange(2) for _ in range(n)]
        expect = max([_lcp(p, q) // b for q in seen], default=0)
        sid = bm.admit(len(p), rnd.randint(0, 5), tokens=p)
        assert bm.reused[sid] == expect
        assert bm.table(sid)[:expect] == [bm.index[tuple(p[: b * (i + 1)])] for i in range(expect)]
        seen.append(p)
        live.append(sid)
        distinct = {tuple(q[: b * k]) for q in seen for k in range(1, len(q) // b + 1)}
        assert bm.stats()["cached"] == len(distinct) and bm.stats()["evictions"] == 0
        _check_invariants(bm)


def test_eviction_is_lru_leaf_first_and_spares_pinned_blocks():
    b = 4
    bm = BlockManager(8, b, prefix_cache=True)
    a_tokens = list(range(16))
    a = bm.admit(16, 0, tokens=a_tokens)  # blocks 0..3, a chain of four
    pinned = bm.admit(8, 0, tokens=[100 + t for t in range(8)])  # blocks 4, 5
    assert bm.table(a) == [0, 1, 2, 3] and bm.table(pinned) == [4, 5]
    bm.free(a)  # cached, idle; released in chain order
    assert bm.stats()["free"] == 2 and bm.available() == 6
    c = bm.admit(16, 0, tokens=[200 + t for t in range(16)])
    # free pages first (6 then 7), then the chain's leaf, then its new leaf
    assert bm.table(c) == [6, 7, 3, 2]
    assert bm.stats()["evictions"] == 2
    assert bm.table(pinned) == [4, 5] and bm.ref[4] == bm.ref[5] == 1
    d = bm.admit(8, 0, tokens=a_tokens[:8])  # A's first two blocks survive
    assert bm.reused[d] == 2 and bm.table(d)[:2] == [0, 1]
    _check_invariants(bm)
    with pytest.raises(PoolExhausted):  # every page is referenced now
        bm.admit(4, 0, tokens=[-5] * 4)


def test_eviction_prefers_least_recently_released():
    bm = BlockManager(4, 4, prefix_cache=True)
    old = bm.admit(4, 0, tokens=[1] * 4)
    new = bm.admit(4, 0, tokens=[2] * 4)
    ob, nb = bm.table(old)[0], bm.table(new)[0]
    bm.free(old)
    bm.free(new)
    bm.admit(8, 0, tokens=[3] * 8)  # two free pages
    sid = bm.admit(4, 0, tokens=[4] * 4)  # evicts one cached page: the older
    assert bm.table(sid) == [ob] and bm.key[nb] == (2,) * 4 and (1,) * 4 not in bm.index
    assert bm.key[ob] == (4,) * 4  # the evicted page now caches the new prompt


def test_hit_on_idle_block_is_not_double_counted():
    """Reusing an idle cached block must not also count it as available."""
    bm = BlockManager(3, 4, prefix_cache=True)
    p = list(range(8))
    bm.free(bm.admit(8, 0, tokens=p))  # two idle cached blocks, one free page
    with pytest.raises(PoolExhausted):  # 2 hits + 2 new pages: only 1 left
        bm.admit(8, 8, tokens=p)
    sid = bm.admit(8, 4, tokens=p)
    assert bm.reused[sid] == 2 and bm.stats()["free"] == 0


def test_token_admission_rules():
    with pytest.raises(InvalidRequest):
        BlockManager(8, 4).admit(4, 0, tokens=[1, 2, 3, 4])  # no prefix cache
    bm = BlockManager(8, 4, prefix_cache=True)
    with pytest.raises(InvalidRequest):
        bm.admit(4, 0, group=0, prefix_len=4, tokens=[1, 2, 3, 4])
    with pytest.raises(InvalidRequest):
        bm.admit(5, 0, tokens=[1, 2, 3, 4])
    assert bm.stats()["seqs"] == 0


# -- incremental allocation, watermark, preemption ------------------------

def test_incremental_admits_more_than_full_reservation(golden):
    g = golden["admission_32L"]
    pool, prompt, out = g["pool_pages"], g["prompt_tokens"], g["output_tokens"]

    def admitted(**kw):
        bm = BlockManager(pool, g["tokens_per_page"], **kw)
        n = 0
        try:
            while True:
                bm.admit(prompt, out)
                n += 1
        except PoolExhausted:
            return n, bm

    full, _ = admitted()
    assert full == g["admitted_isolated"]
    inc, bm = admitted(incremental=True)
    assert inc == pool // g["prompt_only_pages"] == 2
    assert bm.stats()["used"] == 2 * g["prompt_only_pages"]
    held, _ = admitted(incremental=True, watermark=16)
    assert held == 1  # 128 + 16 fit once; a second 128 would leave no headroom


def test_growth_failure_then_preempt_newest_then_resume(golden):
    g = golden["admission_32L"]
    pool, prompt = g["pool_pages"], g["prompt_tokens"]
    bm = BlockManager(pool, 16, incremental=True)
    s0, s1 = bm.admit(prompt, 257), bm.admit(prompt, 257)
    assert bm.num_free == 0
    before = bm.stats(), bm.table(s0), bm.table(s1)
    with pytest.raises(PoolExhausted):  # both need a 129th page now
        bm.prepare_append([s0, s1])
    assert (bm.stats(), bm.table(s0), bm.table(s1)) == before
    victim = bm.newest_running()
    assert victim == s1
    assert bm.preempt(victim) == prompt // 16
    assert bm.context_len(s1) == prompt and bm.table(s1) == []  # keeps its tokens, not its cache
    slots, pairs = bm.prepare_append([s0])
    assert pairs == [] and len(bm.table(s0)) == prompt // 16 + 1
    assert slots == [bm.table(s0)[-1] * 16]
    with pytest.raises(InvalidRequest):  # a preempted sequence takes no step
        bm.prepare_append([s1])
    with pytest.raises(PoolExhausted):  # 128 pages wanted, 127 available
        bm.resume(s1)
    assert bm.stats()["preempted"] == 1
    bm.free(s0)
    bm.resume(s1)
    assert len(bm.table(s1)) == prompt // 16 and bm.context_len(s1) == prompt
    assert len(set(bm.table(s1))) == prompt // 16 and all(bm.ref[x] == 1 for x in bm.table(s1))
    _check_invariants(bm)


def test_watermark_binds_admission_and_resume_not_growth():
    bm = BlockManager(10, 4, incremental=True, watermark=3)
    a = bm.admit(28, 100)  # 7 pages, 3 left = the watermark
    with pytest.raises(PoolExhausted):
        bm.admit(1, 1)
    for _ in range(4 * 3):  # growth may use the headroom
        bm.prepare_append([a])
    assert bm.num_free == 0
    with pytest.raises(PoolExhausted):
        bm.prepare_append([a])
    bm.preempt(a)
    with pytest.raises(PoolExhausted):  # 10 pages + 3 headroom > 10
        bm.resume(a)


def test_full_reservation_never_needs_preemption(golden):
    """A request admitted with its full output allowance reaches that limit
    without taking a page from anyone ("Pick a reservation policy")."""
    g = golden["admission_32L"]
    bm = BlockManager(g["request_pages"], 16)
    s = bm.admit(g["prompt_tokens"], g["output_tokens"])
    for _ in range(g["output_tokens"]):
        bm.prepare_append([s])
    assert bm.num_free == 0 and bm.stats()["used"] == g["request_pages"]


def test_incremental_fork_copies_on_demand():
    bm = BlockManager(6, 4, incremental=True)
    p = bm.admit(6, 10)  # 2 pages, block 1 partial
    (k,) = bm.fork(p, 1)
    assert bm.stats()["spares"] == 0 and bm.ref[bm.table(p)[1]] == 2
    slots, pairs = bm.prepare_append([k, p])
    assert len(pairs) == 1 and pairs[0][0] == bm.table(p)[1]  # the parent writes in place
    assert bm.table(k)[1] == pairs[0][1]
    bm.free(k)
    bm.free(p)
    assert bm.num_free == 6


def test_preempted_prefix_blocks_stay_cached():
    bm = BlockManager(8, 4, incremental=True, prefix_cache=True)
    p = list(range(12))
    s = bm.admit(12, 4, tokens=p)
    bm.preempt(s)
    assert bm.stats()["cached_idle"] == 3
    t = bm.admit(12, 4, tokens=p)  # a recompute of the same prompt could reuse them
    assert bm.reused[t] == 3
    _check_invariants(bm)


@pytest.mark.parametrize("seed", range(16))
def test_random_policies_keep_invariants(seed):
    rnd = random.Random(seed)
    b = rnd.choice([4, 8, 16])
    kw = dict(incremental=rnd.random() < 0.6, watermark=rnd.choice([0, 0, 2, 5]),
              prefix_cache=rnd.random() < 0.6)
    bm = BlockManager(rnd.randint(8, 60), b, **kw)
    vocab = rnd.choice([2, 3])
    prompts = []
    for _ in range(300):
        live = [s for s, q in bm.seqs.items() if q.running]
        stopped = [s for s, q in bm.seqs.items() if not q.running]
        op = rnd.random()
        try:
            if op < 0.25 or not bm.seqs:
                n = rnd.randint(0, 3 * b)
                if kw["prefix_cache"] and rnd.random() < 0.7 and n:
                    if prompts and rnd.random() < 0.6:
                        src = rnd.choice(prompts)
                        p = (src + [rnd.randrange(vocab) for _ in range(n)])[:max(n, 1)]
                    else:
                        p = [rnd.randrange(vocab) for _ in range(n)]
                    prompts.append(p)
                    bm.admit(len(p), rnd.randint(0, 2 * b), tokens=p)
                else:
                    bm.admit(n, rnd.randint(1, 2 * b))
            elif op < 0.35 and live:
                bm.fork(rnd.choice(live), rnd.randint(0, 2))
            elif op < 0.75 and live:
                ids = rnd.sample(live, rnd.randint(1, len(live)))
                before = bm.stats()
                try:
                    bm.prepare_append(ids)
                except PoolExhausted:
                    assert bm.stats() == before
                    bm.preempt(bm.newest_running())
            elif op < 0.85 and stopped:
                bm.resume(rnd.choice(stopped))
            elif op < 0.92 and live:
                bm.preempt(rnd.choice(live))
            elif bm.seqs:
                bm.free(rnd.choice(list(bm.seqs)))
        except (PoolExhausted, InvalidRequest):
            pass
        except Exception as e:  # ReservationExceeded is expected under full reservation
            assert type(e).__name__ == "ReservationExceeded" and not kw["incremental"]
        _check_invariants(bm)
