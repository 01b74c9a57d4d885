"""Pins for the attention oracle: an independent library routine (torch's
scaled_dot_product_attention in float64 on a dense cache), pure-Python brute
force, closed forms and the invariants the pages state (paging changes no
result; shared blocks give identical outputs)."""
import math

import numpy as np
import pytest
import torch

from oracle import paged_attention as pa
from workloads import randn_bf16

B16 = 16


def _dense_case(rng, B, Hq, Hkv, D, ctx, pool_extra=3):
    """Dense per-sequence K/V plus a paged pool holding the same rows at
    randomly chosen physical blocks (the test's own scatter)."""
    ctx = list(ctx)
    nblk = [-(-c // B16) for c in ctx]
    NB = sum(nblk) + pool_extra
    perm = rng.permutation(NB)
    W = max(nblk)
    tables = np.full((B, W), -1, dtype=np.int32)
    kpool = randn_bf16(rng, (NB, Hkv, B16, D))
    vpool = randn_bf16(rng, (NB, Hkv, B16, D))
    dense_k, dense_v = [], []
    off = 0
    for s in range(B):
        tables[s, : nblk[s]] = perm[off : off + nblk[s]]
        off += nblk[s]
        dk = randn_bf16(rng, (Hkv, ctx[s], D))
        dv = randn_bf16(rng, (Hkv, ctx[s], D))
        for t in range(ctx[s]):
            kpool[tables[s, t // B16], :, t % B16, :] = dk[:, t, :]
            vpool[tables[s, t // B16], :, t % B16, :] = dv[:, t, :]
        dense_k.append(dk)
        dense_v.append(dv)
    q = randn_bf16(rng, (B, Hq, D))
    return q, kpool, vpool, tables, np.array(ctx), dense_k, dense_v


def _sdpa_reference(q, dense_k, dense_v, scale):
    B, Hq, D = q.shape
    out = np.zeros((B, Hq, D))
    qt = torch.from_numpy(pa.widen_bf16(q))
    for s in range(B):
        k = torch.from_numpy(pa.widen_bf16(dense_k[s]))
        v = torch.from_numpy(pa.widen_bf16(dense_v[s]))
        G = Hq // k.shape[0]
        k = k.repeat_interleave(G, dim=0)  # query head h uses kv head h // G
        v = v.repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(
            qt[s][:, None, :], k, v, scale=scale)
        out[s] = o[:, 0, :].numpy()
    return out


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (64, 8), (8, 8), (4, 1)])
def test_matches_sdpa_on_dense_cache(Hq, Hkv):
    rng = np.random.default_rng(1)
    ctx = [1, 15, 16, 17, 40, 203]
    q, kp, vp, tab, cl, dk, dv = _dense_case(rng, len(ctx), Hq, Hkv, 128, ctx)
    scale = 1 / math.sqrt(128)
    got = pa.paged_decode_attention(q, kp, vp, tab, cl, scale)
    ref = _sdpa_reference(q, dk, dv, scale)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_identity_table_is_contiguous_cache():
    # Identity table: block i of sequence s is physical block s*W + i, so the
    # pool read in order is the contiguous (base + stride*t) cache.
    rng = np.random.default_rng(2)
    B, Hq, Hkv, D, W = 3, 8, 2, 128, 4
    kp = randn_bf16(rng, (B * W, Hkv, B16, D))
    vp = randn_bf16(rng, (B * W, Hkv, B16, D))
    q = randn_bf16(rng, (B, Hq, D))
    tab = np.arange(B * W, dtype=np.int32).reshape(B, W)
    ctx = np.array([64, 33, 7])
    got = pa.paged_decode_attention(q, kp, vp, tab, ctx, 0.1)
    dk = [kp[s * W:(s + 1) * W].transpose(1, 0, 2, 3).reshape(Hkv, W * B16, D)[:, : ctx[s]] for s in range(B)]
    dv = [vp[s * W:(s + 1) * W].transpose(1, 0, 2, 3).reshape(Hkv, W * B16, D)[:, : ctx[s]] for s in range(B)]
    np.testing.assert_allclose(got, _sdpa_reference(q, dk, dv, 0.1), rtol=0, atol=1e-12)


def test_brute_force_pure_python():
    rng = np.random.default_rng(3)
    B, Hq, Hkv, D = 2, 4, 2, 4
    ctx = [5, 20]
    q, kp, vp, tab, cl, _, _ = _dense_case(rng, B, Hq, Hkv, D, ctx)
    scale = 0.7
    got = pa.paged_decode_attention(q, kp, vp, tab, cl, scale)

    def f(bits):
        return float(pa.widen_bf16(np.array([bits], dtype=np.uint16))[0])

    for s in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            xs, rows = [], []
            for t in range(ctx[s]):
                blk, r = int(tab[s][t // 16]), t % 16
                xs.append(scale * sum(f(q[s, h, d]) * f(kp[blk, g, r, d]) for d in range(D)))
                rows.append([f(vp[blk, g, r, d]) for d in range(D)])
            m = max(xs)
            ws = [math.exp(x - m) for x in xs]
            den = sum(ws)
            for d in range(D):
                exp_val = sum(w * row[d] for w, row in zip(ws, rows)) / den
                assert abs(got[s, h, d] - exp_val) < 1e-12


def test_permutation_of_physical_blocks_is_invisible():
    rng = np.random.default_rng(4)
    ctx = [3, 50, 129]
    q, kp, vp, tab, cl, _, _ = _dense_case(rng, 3, 32, 8, 128, ctx)
    base = pa.paged_decode_attention(q, kp, vp, tab, cl, 0.088)
    NB = kp.shape[0]
    perm = rng.permutation(NB)  # physical block b moves to perm[b]
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    kp2[perm], vp2[perm] = kp, vp
    tab2 = np.where(tab >= 0, perm[np.maximum(tab, 0)], -1).astype(np.int32)
    moved = pa.paged_decode_attention(q, kp2, vp2, tab2, cl, 0.088)
    assert np.array_equal(base, moved)


def test_shared_blocks_give_identical_outputs():
    rng = np.random.default_rng(5)
    q, kp, vp, tab, cl, _, _ = _dense_case(rng, 1, 32, 8, 128, [77])
    q2 = np.concatenate([q, q])
    tab2 = np.concatenate([tab, tab])
    out = pa.paged_decode_attention(q2, kp, vp, tab2, np.array([77, 77]), 0.088)
    assert np.array_equal(out[0], out[1])


def test_single_token_returns_its_value():
    rng = np.random.default_rng(6)
    q, kp, vp, tab, cl, _, dv = _dense_case(rng, 1, 32, 8, 128, [1])
    out = pa.paged_decode_attention(q, kp, vp, tab, cl, 0.088)
    for h in range(32):
        assert np.array_equal(out[0, h], pa.widen_bf16(dv[0][h // 4, 0]))


def test_equal_keys_average_the_values():
    rng = np.random.default_rng(7)
    q, kp, vp, tab, cl, _, dv = _dense_case(rng, 1, 8, 2, 128, [37])
    kp[:] = kp[tab[0, 0], :, 0:1, :]  # every key equal to one row
    out = pa.paged_decode_attention(q, kp, vp, tab, cl, 0.3)
    for h in range(8):
        mean = pa.widen_bf16(dv[0][h // 4]).mean(axis=0)
        np.testing.assert_allclose(out[0, h], mean, rtol=0, atol=1e-14)


def test_two_token_weights_and_no_overflow():
    # k0 = e0 + e1, k1 = e1, v0 = 1, v1 = 0.
    D = 128
    one = np.uint16(0x3F80)  # bf16 1.0
    kp = np.zeros((1, 1, B16, D), dtype=np.uint16)
    vp = np.zeros((1, 1, B16, D), dtype=np.uint16)
    kp[0, 0, 0, 0] = one
    kp[0, 0, 0, 1] = one
    kp[0, 0, 1, 1] = one
    vp[0, 0, 0, :] = one
    tab, ctx = np.array([[0]]), np.array([2])
    # q = e0, scale = ln 3: logits ln 3 and 0, weights 3/4 and 1/4.
    q = np.zeros((1, 1, D), dtype=np.uint16)
    q[0, 0, 0] = one
    out = pa.paged_decode_attention(q, kp, vp, tab, ctx, math.log(3.0))
    np.testing.assert_allclose(out[0, 0], 0.75, rtol=0, atol=1e-12)
    # q = e0 + 1000 e1, scale 1: logits 1001 and 1000 (exp overflows without
    # the max shift), weights e/(e+1) and 1/(e+1).
    q[0, 0, 1] = np.uint16(0x447A)  # bf16 1000.0
    out = pa.paged_decode_attention(q, kp, vp, tab, ctx, 1.0)
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out[0, 0], math.e / (math.e + 1.0), rtol=0, atol=1e-12)


def test_gqa_head_mapping():
    # Each KV head's values are constant c_g, so head h must return c_{h // G}.
    rng = np.random.default_rng(8)
    Hq, Hkv, D = 16, 4, 128
    q, kp, vp, tab, cl, _, _ = _dense_case(rng, 2, Hq, Hkv, D, [20, 45])
    consts = [0x3F80, 0x4000, 0x4040, 0x4080]  # 1, 2, 3, 4
    for g in range(Hkv):
        vp[:, g] = consts[g]
    out = pa.paged_decode_attention(q, kp, vp, tab, cl, 0.088)
    for h in range(Hq):
        np.testing.assert_allclose(out[:, h], float(h // (Hq // Hkv) + 1), atol=1e-12)


def test_zero_context_is_zero():
    rng = np.random.default_rng(9)
    q, kp, vp, tab, cl, _, _ = _dense_case(rng, 2, 8, 2, 128, [5, 9])
    out = pa.paged_decode_attention(q, kp, vp, tab, np.array([0, 9]), 0.1)
    assert not out[0].any()


def test_slots_past_context_are_ignored():
    rng = np.random.default_rng(10)
    q, kp, vp, tab, cl, _, _ = _dense_case(rng, 2, 8, 2, 128, [5, 19])
    base = pa.paged_decode_attention(q, kp, vp, tab, cl, 0.1)
    kp2, vp2 = kp.copy(), vp.copy()
    kp2[tab[0, 0], :, 5:] = 0x7FC0  # NaN past ctx
    vp2[tab[0, 0], :, 5:] = 0x7FC0
    kp2[tab[1, 1], :, 3:] = 0x7FC0
    vp2[tab[1, 1], :, 3:] = 0x7FC0
    assert np.array_equal(base, pa.paged_decode_attention(q, kp2, vp2, tab, cl, 0.1))


@pytest.mark.parametrize("P", [16, 32, 48, 1000])
def test_partitioned_equals_direct(P):
    rng = np.random.default_rng(11)
    q, kp, vp, tab, cl, _, _ = _dense_case(rng, 3, 16, 4, 128, [1, 90, 203])
    a = pa.paged_decode_attention(q, kp, vp, tab, cl, 0.088)
    b = pa.partitioned_decode_attention(q, kp, vp, tab, cl, 0.088, P)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)
