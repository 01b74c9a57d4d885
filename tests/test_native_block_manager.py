"""The C++ block manager against the oracle's: the pages' worked numbers and
bit-exact agreement (block ids, slots, copy pairs, refcounts, errors) over
random operation sequences and the synthetic workloads' events. CPU only."""
import random
import threading

import pytest

from oracle import block_manager as obm
from workloads import make_workload


@pytest.fixture(scope="module")
def nat():
    from tests.conftest import build_native
    build_native()
    import paged_kv_cache_49_gb300._native as n
    return n


def test_worked_admission_numbers(nat, golden):
    g = golden["admission_32L"]
    bm = nat.BlockManager(g["pool_pages"])
    for _ in range(7):
        bm.admit(g["prompt_tokens"], g["output_tokens"], 0, g["prompt_tokens"])
    st = bm.stats()
    assert st["used"] == g["seven_shared_pages"] and st["free"] == g["seven_shared_free_after"]
    with pytest.raises(nat.PoolExhausted):
        bm.admit(g["prompt_tokens"], g["output_tokens"], 0, g["prompt_tokens"])
    assert bm.stats() == st
    iso = nat.BlockManager(g["pool_pages"])
    iso.admit(g["prompt_tokens"], g["output_tokens"], 0, g["prompt_tokens"])
    assert iso.stats()["used"] == g["request_pages"]
    with pytest.raises(nat.PoolExhausted):
        iso.admit(g["prompt_tokens"], g["output_tokens"], 1, g["prompt_tokens"])


def test_fanout_numbers(nat, golden):
    g = golden["fanout_n8"]
    bm = nat.BlockManager(4096)
    p = bm.admit(g["prompt_tokens"], g["output_tokens"])
    bm.fork(p, g["samples"] - 1)
    assert bm.stats()["used"] * 16 == g["shared_tokens"]


def _err_kind(nat, e):
    if isinstance(e, (nat.PoolExhausted, obm.PoolExhausted)):
        return "nomem"
    if isinstance(e, (nat.ReservationExceeded, obm.ReservationExceeded)):
        return "nospc"
    return "inval"


def _both(nat, fa, fb):
    ra = rb = ea = eb = None
    try:
        ra = fa()
    except (obm.BlockManagerError,) as e:
        ea = _err_kind(nat, e)
    try:
        rb = fb()
    except nat.PkvError as e:
        eb = _err_kind(nat, e)
    assert ea == eb
    assert ra == rb
    return ra


def _same_state(o, n, ids):
    assert o.stats() == n.stats()
    for s in ids:
        assert o.table(s) == n.table(s)
        assert o.context_len(s) == n.context_len(s)
    for b in range(o.num_blocks):
        assert o.ref[b] == n.refcount(b)


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("bt", [16, 8, 32, 64])
def test_random_operations_match_oracle(nat, seed, bt):
    rnd = random.Random(seed)
    nb = rnd.randint(16, 160) * 16 // bt
    order = rnd.sample(range(nb), nb) if seed % 2 else None
    o = obm.BlockManager(nb, bt, order)
    n = nat.BlockManager(nb, bt, order)
    for _ in range(250):
        live = sorted(o.seqs)
        op = rnd.random()
        if op < 0.3 or not live:
            grp = rnd.choice([-1, -1, 0, 1])
            p = rnd.randint(0, 60)
            args = (p, rnd.randint(0, 40), grp, bt * rnd.randint(0, p // bt) if grp >= 0 else 0)
            _both(nat, lambda: o.admit(*args), lambda: n.admit(*args))
        elif op < 0.45:
            par, k = rnd.choice(live), rnd.randint(0, 3)
            _both(nat, lambda: o.fork(par, k), lambda: n.fork(par, k))
        elif op < 0.85:
            ids = rnd.sample(live, rnd.randint(1, len(live)))
            _both(nat, lambda: o.prepare_append(ids), lambda: n.prepare_append(ids))
        elif op < 0.95:
            s = rnd.choice(live)
            _both(nat, lambda: o.free(s), lambda: n.free(s))
        else:  # invalid calls
            _both(nat, lambda: o.free(10 ** 6), lambda: n.free(10 ** 6))
            if live:
                _both(nat, lambda: o.prepare_append([live[0], live[0]]),
                      lambda: n.prepare_append([live[0], live[0]]))
        _same_state(o, n, sorted(o.seqs))


@pytest.mark.parametrize("name", ["tiny", "tiny_nan", "prefix_admission", "fanout", "llama3_8b_b64"])
def test_workload_events_match_oracle(nat, name):
    w = make_workload(name)
    o = obm.BlockManager(w.pool_blocks, 16, w.free_order)
    n = nat.BlockManager(w.pool_blocks, 16, w.free_order)
    for ev in w.events:
        if ev[0] == "admit":
            _both(nat, lambda: o.admit(*ev[1:]), lambda: n.admit(*ev[1:]))
        elif ev[0] == "fork":
            _both(nat, lambda: o.fork(ev[1], ev[2]), lambda: n.fork(ev[1], ev[2]))
        else:
            counts = ev[1]
            ids = sorted(counts)
            for t in range(max(counts.values()) if counts else 0):
                batch = [s for s in ids if counts[s] > t]
                _both(nat, lambda: o.prepare_append(batch), lambda: n.prepare_append(batch))
    _both(nat, lambda: o.prepare_append(w.batch), lambda: n.prepare_append(w.batch))
    _same_state(o, n, w.batch)
    width = max(len(o.table(s)) for s in w.batch)
    tables, ctx = n.batch_tables(w.batch, width)
    for i, s in enumerate(w.batch):
        t = o.table(s)
        assert tables[i, : len(t)].tolist() == t and (tables[i, len(t):] == -1).all()
        assert int(ctx[i]) == o.context_len(s)


def test_concurrent_admissions_never_overcommit(nat):
    # "Reserve the page a request has not written yet": two admissions that
    # read the same free count must not both succeed past the pool.
    bm = nat.BlockManager(256)
    admitted, lock = [], threading.Lock()

    def worker():
        for _ in range(20):
            try:
                sid = bm.admit(2048, 257)
                with lock:
                    admitted.append(sid)
            except nat.PoolExhausted:
                pass

    threads = [threading.Thread(target=worker) for _ in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert len(admitted) == 1 and bm.stats()["used"] == 145


def _same_policy_state(nat, o, n):
    assert o.stats() == n.stats()
    for s in sorted(o.seqs):
        assert o.table(s) == n.table(s)
        assert o.context_len(s) == n.context_len(s)
    for b in range(o.num_blocks):
        assert o.ref[b] == n.refcount(b)
    assert o.newest_running() == n.newest_running()
    for s in sorted(o.seqs):
        if o.seqs[s].running:
            cap = len(o.table(s)) * o.b
            assert o.slots(s, 0, cap) == n.slots(s, 0, cap)
            _both(nat, lambda: o.slots(s, 1, cap), lambda: n.slots(s, 1, cap))  # one past the table


@pytest.mark.parametrize("seed", range(10))
@pytest.mark.parametrize("incremental,watermark,prefix_cache",
                         [(True, 0, False), (True, 3, False), (False, 0, True), (True, 2, True)])
def test_random_policies_match_oracle(nat, seed, incremental, watermark, prefix_cache):
    """Incremental growth, watermark, preemption, resume and prefix-cache hits
    and evictions decided identically (block ids included) by both managers."""
    rnd = random.Random(1000 + seed)
    bt = rnd.choice([8, 16])
    nb = rnd.randint(6, 40)
    order = rnd.sample(range(nb), nb) if seed % 2 else None
    kw = dict(incremental=incremental, watermark=watermark, prefix_cache=prefix_cache)
    o = obm.BlockManager(nb, bt, order, **kw)
    n = nat.BlockManager(nb, bt, order, **kw)
    prompts = []
    for _ in range(300):
        running = [s for s, q in o.seqs.items() if q.running]
        stopped = [s for s, q in o.seqs.items() if not q.running]
        op = rnd.random()
        if op < 0.25 or not o.seqs:
            plen = rnd.randint(0, 4 * bt)
            if prefix_cache and plen and rnd.random() < 0.7:
                if prompts and rnd.random() < 0.6:
                    src = rnd.choice(prompts)
                    keep = len(src) if rnd.random() < 0.5 else rnd.randint(0, len(src))
                    p = (src[:keep] + [rnd.randrange(2) for _ in range(plen)])[:plen]
                else:
                    p = [rnd.randrange(2) for _ in range(plen)]
                prompts.append(p)
                args = (plen, rnd.randint(0, 2 * bt))
                sid = _both(nat, lambda: o.admit(*args, tokens=p), lambda: n.admit(*args, tokens=p))
                if sid is not None:
                    assert o.reused[sid] == n.reused[sid]
            else:
                grp = rnd.choice([-1, -1, 0])
                args = (plen, rnd.randint(1, 2 * bt), grp, bt * rnd.randint(0, plen // bt) if grp >= 0 else 0)
                _both(nat, lambda: o.admit(*args), lambda: n.admit(*args))
        elif op < 0.35 and running:
            par, k = rnd.choice(running), rnd.randint(0, 2)
            _both(nat, lambda: o.fork(par, k), lambda: n.fork(par, k))
        elif op < 0.75 and running:
            ids = rnd.sample(running, rnd.randint(1, len(running)))
            r = _both(nat, lambda: o.prepare_append(ids), lambda: n.prepare_append(ids))
            if r is None and incremental:  # refused: preempt the newest and go on
                v = o.newest_running()
                assert _both(nat, lambda: o.preempt(v), lambda: n.preempt(v)) is not None
        elif op < 0.85 and stopped:
            s = rnd.choice(stopped)
            _both(nat, lambda: o.resume(s), lambda: n.resume(s))
        elif op < 0.9 and running:
            s = rnd.choice(running)
            _both(nat, lambda: o.preempt(s), lambda: n.preempt(s))
        elif op < 0.97 and o.seqs:
            s = rnd.choice(sorted(o.seqs))
            _both(nat, lambda: o.free(s), lambda: n.free(s))
        else:  # invalid calls
            if stopped:
                s = stopped[0]
                _both(nat, lambda: o.prepare_append([s]), lambda: n.prepare_append([s]))
                _both(nat, lambda: o.fork(s, 1), lambda: n.fork(s, 1))
                _both(nat, lambda: o.preempt(s), lambda: n.preempt(s))
            if running:
                s = running[0]
                _both(nat, lambda: o.resume(s), lambda: n.resume(s))
        _same_policy_state(nat, o, n)


def test_prefix_hit_worked_example_native(nat, golden):
    g = golden["prefix_hit_8000"]
    rnd = random.Random(0)
    cached = [rnd.randrange(32000) for _ in range(g["matching_tokens"] + 200)]
    bm = nat.BlockManager(2048, g["block_tokens"], prefix_cache=True)
    first = bm.admit(len(cached), 1, tokens=cached)
    req = list(cached)
    req[g["matching_tokens"]] += 1
    sid = bm.admit(len(req), 1, tokens=req)
    assert bm.reused[sid] == g["reused_blocks"]
    assert bm.table(sid)[: g["reused_blocks"]] == bm.table(first)[: g["reused_blocks"]]
    with pytest.raises(nat.PkvError):  # tokens need a prefix-cache manager
        nat.BlockManager(64).admit(4, 1, tokens=[1, 2, 3, 4])


def test_incremental_admission_and_preemption_native(nat, golden):
    g = golden["admission_32L"]
    bm = nat.BlockManager(g["pool_pages"], incremental=True)
    s0 = bm.admit(g["prompt_tokens"], g["output_tokens"])
    s1 = bm.admit(g["prompt_tokens"], g["output_tokens"])
    with pytest.raises(nat.PoolExhausted):
        bm.admit(g["prompt_tokens"], g["output_tokens"])
    with pytest.raises(nat.PoolExhausted):
        bm.prepare_append([s0, s1])
    assert bm.newest_running() == s1 and bm.preempt(s1) == g["prompt_only_pages"]
    bm.prepare_append([s0])
    assert bm.stats()["preempted"] == 1 and bm.context_len(s1) == g["prompt_tokens"]
    with pytest.raises(nat.PoolExhausted):
        bm.resume(s1)
    bm.free(s0)
    bm.resume(s1)
    assert len(bm.table(s1)) == g["prompt_only_pages"]
    held = nat.BlockManager(g["pool_pages"], incremental=True, watermark=16)
    held.admit(g["prompt_tokens"], g["output_tokens"])
    with pytest.raises(nat.PoolExhausted):
        held.admit(g["prompt_tokens"], g["output_tokens"])
