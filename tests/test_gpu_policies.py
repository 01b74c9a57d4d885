"""The block manager's incremental, preemption and prefix-cache decisions
driving the CUDA path (append kernel and decode attention through the C ABI).

Each token position's K/V is a seeded function of the token prefix that ends
there, as a model's KV is. A sequence's attention through its block table --
blocks reused from the prefix cache, pages recycled by eviction or after a
preemption -- must equal the oracle's attention over the K/V its own tokens
define (max |err| 2e-2, mean |err| 2e-3), and a recomputed sequence must
reproduce its pre-preemption output bit for bit.
"""
import zlib

import numpy as np
import pytest
import torch

from oracle import paged_attention as pa
from workloads import randn_bf16

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3
HQ, HKV, D = 8, 2, 128


@pytest.fixture(scope="module")
def pkv():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tests.conftest import build_native
    build_native()
    import paged_kv_cache_49_gb300 as m
    return m


def _kv_at(tokens, t):
    """bf16 bits [2, HKV, D]: K and V of position t, seeded by tokens[:t+1]."""
    seed = zlib.crc32(np.asarray(tokens[: t + 1], dtype=np.int64).tobytes())
    return randn_bf16(np.random.default_rng(seed), (2, HKV, D))


def _kv_rows(tokens, first, n):
    rows = np.stack([_kv_at(tokens, t) for t in range(first, first + n)])  # [n, 2, HKV, D]
    return rows[:, 0], rows[:, 1]


def _write(pkv, eng, sid, tokens, first, n):
    k, v = _kv_rows(tokens, first, n)
    eng.write_positions(sid, first, pkv.bf16_from_bits(k).cuda(), pkv.bf16_from_bits(v).cuda())


def _attend(pkv, eng, sids, q_bits, scale):
    tables, ctx = eng.bm.batch_tables(sids, max(len(eng.bm.table(s)) for s in sids))
    q = pkv.bf16_from_bits(q_bits).cuda()
    out = torch.empty_like(q)
    ws = pkv.AttentionWorkspace(len(sids), HKV)
    pkv.attn_decode(q, eng.k_cache, eng.v_cache, tables.cuda(), ctx.cuda(), scale, out, ws)
    torch.cuda.synchronize()
    assert eng.read_errors() == 0 and ws.read_error() == 0
    return out


def _oracle(q_bits, token_lists, scale, b):
    """Attention over each sequence's own K/V, laid out contiguously."""
    n = len(token_lists)
    width = max(-(-len(t) // b) for t in token_lists)
    kc = np.zeros((n * width, HKV, b, D), np.uint16)
    vc = np.zeros_like(kc)
    tables = np.arange(n * width, dtype=np.int64).reshape(n, width)
    for i, toks in enumerate(token_lists):
        k, v = _kv_rows(toks, 0, len(toks))
        for t in range(len(toks)):
            kc[tables[i, t // b], :, t % b] = k[t]
            vc[tables[i, t // b], :, t % b] = v[t]
    ctx = np.array([len(t) for t in token_lists])
    return pa.paged_decode_attention(q_bits, kc, vc, tables, ctx, scale)


def _close(out, ref):
    g = out.float().cpu().numpy().astype(np.float64)
    d = np.abs(g - ref)
    assert np.isfinite(g).all() and d.max() <= MAX_ABS and d.mean() <= MEAN_ABS, (d.max(), d.mean())


@pytest.mark.parametrize("b", [16, 8])
def test_prefix_cache_reuse_and_eviction(pkv, b):
    rnd = np.random.default_rng(7)
    scale = D ** -0.5
    eng = pkv.PagedKVEngine(40, HQ, HKV, D, block_tokens=b, prefix_cache=True)
    system = rnd.integers(0, 32000, 5 * b + 3).tolist()
    a_toks = system + rnd.integers(0, 32000, 2 * b).tolist()
    a = eng.bm.admit(len(a_toks), b, tokens=a_toks)
    _write(pkv, eng, a, a_toks, 0, len(a_toks))
    c_toks = system + rnd.integers(0, 32000, b + 5).tolist()
    c = eng.bm.admit(len(c_toks), b, tokens=c_toks)
    reused = eng.bm.reused[c]
    assert reused == len(system) // b
    _write(pkv, eng, c, c_toks, reused * b, len(c_toks) - reused * b)  # only the uncached suffix
    q = randn_bf16(np.random.default_rng(1), (2, HQ, D))
    _close(_attend(pkv, eng, [a, c], q, scale), _oracle(q, [a_toks, c_toks], scale, b))
    # release both; fill the pool with other prompts so eviction recycles cached pages
    eng.bm.free(a)
    eng.bm.free(c)
    others, live = [], []
    while eng.bm.stats()["available"] >= 4:
        toks = rnd.integers(0, 32000, 3 * b).tolist()
        sid = eng.bm.admit(len(toks), 0, tokens=toks)
        _write(pkv, eng, sid, toks, 0, len(toks))
        others.append(toks)
        live.append(sid)
    assert eng.bm.stats()["evictions"] > 0
    for sid in live[: len(live) // 2]:
        eng.bm.free(sid)
    d_toks = system + rnd.integers(0, 32000, 7).tolist()
    dd = eng.bm.admit(len(d_toks), 1, tokens=d_toks)
    r = eng.bm.reused[dd]
    _write(pkv, eng, dd, d_toks, r * b, len(d_toks) - r * b)
    rest = live[len(live) // 2:]
    q = randn_bf16(np.random.default_rng(2), (1 + len(rest), HQ, D))
    out = _attend(pkv, eng, [dd] + rest, q, scale)
    _close(out, _oracle(q, [d_toks] + others[len(live) // 2:], scale, b))


def test_preempt_resume_recompute_is_exact(pkv):
    b, scale = 16, D ** -0.5
    rnd = np.random.default_rng(3)
    eng = pkv.PagedKVEngine(24, HQ, HKV, D, incremental=True)
    toks = [rnd.integers(0, 32000, n).tolist() for n in (70, 90, 100)]
    sids = [eng.bm.admit(len(t), 64) for t in toks]
    for sid, t in zip(sids, toks):
        _write(pkv, eng, sid, t, 0, len(t))
    # decode until a step cannot get its pages
    while True:
        running = [s for s in sids if eng.bm.table(s)]
        nxt = [rnd.integers(0, 32000) for _ in running]
        try:
            slots, pairs = eng.bm.prepare_append(running)
        except pkv.PoolExhausted:
            break
        assert pairs == []
        for s, x in zip(running, nxt):
            toks[sids.index(s)].append(int(x))
        kv = [_kv_at(toks[sids.index(s)], eng.bm.context_len(s) - 1) for s in running]
        k = pkv.bf16_from_bits(np.stack([x[0] for x in kv])).cuda()
        v = pkv.bf16_from_bits(np.stack([x[1] for x in kv])).cuda()
        pkv.append(k, v, torch.tensor(slots, dtype=torch.int64).cuda(), eng.k_cache, eng.v_cache, eng.error)
    victim = eng.bm.newest_running()
    vi = sids.index(victim)
    q = randn_bf16(np.random.default_rng(4), (1, HQ, D))
    before = _attend(pkv, eng, [victim], q, scale).clone()
    _close(before, _oracle(q, [toks[vi]], scale, b))
    old_pages = eng.bm.table(victim)
    eng.bm.preempt(victim)
    # the survivors grow into the freed pages, overwriting the victim's KV
    survivors = [s for s in sids if s != victim]
    for _ in range(b):
        slots, _ = eng.bm.prepare_append(survivors)
        for s in survivors:
            toks[sids.index(s)].append(int(rnd.integers(0, 32000)))
        kv = [_kv_at(toks[sids.index(s)], eng.bm.context_len(s) - 1) for s in survivors]
        k = pkv.bf16_from_bits(np.stack([x[0] for x in kv])).cuda()
        v = pkv.bf16_from_bits(np.stack([x[1] for x in kv])).cuda()
        pkv.append(k, v, torch.tensor(slots, dtype=torch.int64).cuda(), eng.k_cache, eng.v_cache, eng.error)
    assert set(old_pages) & {x for s in survivors for x in eng.bm.table(s)}
    while True:  # make room: end survivors until the victim fits again
        try:
            eng.bm.resume(victim)
            break
        except pkv.PoolExhausted:
            eng.bm.free(survivors.pop(0))
    assert eng.bm.context_len(victim) == len(toks[vi])
    _write(pkv, eng, victim, toks[vi], 0, len(toks[vi]))  # the recompute
    after = _attend(pkv, eng, [victim], q, scale)
    assert torch.equal(before, after)
    rows = [survivors[0]] if survivors else []
    if rows:
        q2 = randn_bf16(np.random.default_rng(5), (2, HQ, D))
        _close(_attend(pkv, eng, [victim] + rows, q2, scale),
               _oracle(q2, [toks[vi], toks[sids.index(rows[0])]], scale, b))
