"""Pins for the oracle's slot arithmetic, append and block copy."""
import numpy as np

from oracle import cache_ops, paged_attention as pa
from workloads import randn_bf16


def test_identity_table_slot_is_position():
    # A contiguous cache addresses token t at base + stride * t ("KV cache
    # systems", block-table paragraph); with the identity table the slot is t.
    table = np.arange(64)
    for t in range(1024):
        assert cache_ops.slot_of(table, t) == t


def test_slot_follows_the_table():
    table = np.array([7, 3, 11])
    assert [cache_ops.slot_of(table, t) for t in (0, 15, 16, 31, 32, 47)] == [112, 127, 48, 63, 176, 191]


def test_append_round_trips_through_the_gather():
    rng = np.random.default_rng(0)
    NB, Hkv, D = 10, 4, 128
    kc = randn_bf16(rng, (NB, Hkv, 16, D))
    vc = randn_bf16(rng, (NB, Hkv, 16, D))
    before_k, before_v = kc.copy(), vc.copy()
    table = np.array([6, 2, 9])
    positions = [0, 17, 40]
    k_new = randn_bf16(rng, (3, Hkv, D))
    v_new = randn_bf16(rng, (3, Hkv, D))
    slots = [cache_ops.slot_of(table, p) for p in positions]
    cache_ops.append_kv(kc, vc, k_new, v_new, slots)
    for i, p in enumerate(positions):
        for g in range(Hkv):
            got_k = pa.gather_tokens(kc, table, p + 1, g)[p]
            assert np.array_equal(got_k, pa.widen_bf16(k_new[i, g]))
            assert np.array_equal(pa.gather_tokens(vc, table, p + 1, g)[p], pa.widen_bf16(v_new[i, g]))
    changed = np.argwhere((kc != before_k).any(axis=-1))
    assert {(int(b), int(r)) for b, _, r in changed} <= {(6, 0), (2, 1), (9, 8)}
    assert int((vc != before_v).any(axis=-1).sum()) <= 3 * Hkv


def test_negative_slot_writes_nothing():
    rng = np.random.default_rng(1)
    kc = randn_bf16(rng, (4, 2, 16, 8))
    vc = randn_bf16(rng, (4, 2, 16, 8))
    k0, v0 = kc.copy(), vc.copy()
    cache_ops.append_kv(kc, vc, randn_bf16(rng, (2, 2, 8)), randn_bf16(rng, (2, 2, 8)), [-1, -7])
    assert np.array_equal(kc, k0) and np.array_equal(vc, v0)


def test_copy_blocks_copies_whole_blocks_only():
    rng = np.random.default_rng(2)
    kc = randn_bf16(rng, (8, 4, 16, 128))
    vc = randn_bf16(rng, (8, 4, 16, 128))
    k0, v0 = kc.copy(), vc.copy()
    cache_ops.copy_blocks(kc, vc, [(1, 5), (3, 6)])
    assert np.array_equal(kc[5], k0[1]) and np.array_equal(vc[6], v0[3])
    untouched = [0, 1, 2, 3, 4, 7]
    assert np.array_equal(kc[untouched], k0[untouched]) and np.array_equal(vc[untouched], v0[untouched])


def test_copy_blocks_reads_sources_before_writing():
    rng = np.random.default_rng(3)
    kc = randn_bf16(rng, (4, 1, 16, 8))
    vc = randn_bf16(rng, (4, 1, 16, 8))
    a_k, a_v = kc.copy(), vc.copy()
    b_k, b_v = kc.copy(), vc.copy()
    cache_ops.copy_blocks(a_k, a_v, [(0, 1), (1, 2)])
    cache_ops.copy_blocks(b_k, b_v, [(1, 2), (0, 1)])
    assert np.array_equal(a_k, b_k) and np.array_equal(a_v, b_v)
    assert np.array_equal(a_k[2], kc[1])
