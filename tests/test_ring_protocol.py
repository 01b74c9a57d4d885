"""The decode kernel's stage ring as a protocol, under random schedules.

Each stage of the ring has a full and an empty mbarrier; a copy into stage
j % 8 waits on the empty barrier's phase for the release of tile j - 8 with a
parity wait, which passes whenever the barrier's completed-phase count has
the other parity -- so it is right only while the barrier is at most one
phase short of the one waited for. The merge warp copies the first piece's
first tiles (at most a ring's depth, all at once) and the producer the rest.
This host model checks that the scheme never fills a stage whose previous
tile is unread and never lets a consumer read a stale stage, with copies
landing out of order, and that letting the merge warp copy more than a
ring's depth while the producer runs ahead does break it."""
import random

K = 8  # stages


class Bar:
    def __init__(self):
        self.k = 0  # completed phases

    def try_wait(self, parity):
        return (self.k & 1) != parity


def run(n, total, seed):
    """Tiles [0, n) copied by the merge warp, [n, total) by the producer;
    consumer warp w takes tiles w, w + 4, ...; returns the violations."""
    rnd = random.Random(seed)
    full = [Bar() for _ in range(K)]
    empty = [Bar() for _ in range(K)]
    content = [None] * K
    released = set()
    inflight = []
    errors = []

    def issue(j):
        if j >= K and (j - K) not in released:
            errors.append(f"tile {j} copied before tile {j - K} was released")
        inflight.append((j % K, j))

    def issuer(lo, hi, at_once):
        for j in range(lo, hi):
            if not (at_once and j < K):
                while not empty[j % K].try_wait(((j // K) & 1) ^ 1):
                    yield
            issue(j)
            yield

    def consumer(w):
        for g in range(w, total, 4):
            st = g % K
            while not full[st].try_wait((g // K) & 1):
                yield
            if content[st] != g:
                errors.append(f"tile {g} read from a stage holding {content[st]}")
            yield
            released.add(g)
            empty[st].k += 1
            yield

    def copy_engine():
        while True:
            if inflight:
                st, j = inflight.pop(rnd.randrange(len(inflight)))
                content[st] = j
                full[st].k += 1
            yield

    agents = [issuer(0, n, True), issuer(n, total, False)] + [consumer(w) for w in range(4)]
    engine = copy_engine()
    for _ in range(300000):
        if not agents or errors:
            break
        a = rnd.choice(agents + [engine, engine])
        try:
            next(a)
        except StopIteration:
            agents.remove(a)
    return errors or (["did not finish"] if agents else [])


def test_first_ring_full_from_a_second_issuer_is_safe():
    for seed in range(600):
        r = random.Random(seed)
        n = r.randint(0, K)
        total = n + r.randint(0, 70)
        assert run(n, total, seed) == [], (n, total, seed)


def test_a_longer_early_range_breaks_the_parity_waits():
    bad = 0
    for seed in range(200):
        r = random.Random(seed)
        n = r.randint(3 * K, 60)
        if run(n, n + 40, seed):
            bad += 1
    assert bad > 0
