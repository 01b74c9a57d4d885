"""Batches past the size at which two merge slots still leave two CTAs per
SM (about 2,100 sequences): the kernel then runs its one-merge-slot
instantiations -- for 16-token blocks, for 8-, 32- and 64-token blocks, and
for cascade attention's private pass. Each is checked against the oracle on
a sample of rows (the oracle is a plain loop), including empty contexts."""
import numpy as np
import pytest
import torch

from oracle import paged_attention as pa
from workloads import randn_bf16

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3


@pytest.fixture(scope="module")
def pkv():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tests.conftest import build_native
    build_native()
    import paged_kv_cache_49_gb300 as m
    return m


def _batch(rng, ctx, bt, hq, hkv, d=128, shared=None):
    """Tables over a permuted pool for contexts `ctx`; `shared` = (members,
    blocks) lists whose members share their first `blocks` blocks."""
    B = len(ctx)
    nblk = [-(-int(c) // bt) for c in ctx]
    width = max(1, max(nblk))
    total = sum(nblk) + 8
    perm = rng.permutation(total).astype(np.int32)
    tables = np.full((B, width), -1, np.int32)
    nxt = 0
    first = {}
    for members, blocks in shared or []:
        ids = perm[nxt:nxt + blocks]
        nxt += blocks
        for m in members:
            first[m] = ids
    for s in range(B):
        start = 0
        if s in first:
            tables[s, :len(first[s])] = first[s]
            start = len(first[s])
        for j in range(start, nblk[s]):
            tables[s, j] = perm[nxt]
            nxt += 1
    kc = randn_bf16(rng, (total, hkv, bt, d))
    vc = randn_bf16(rng, (total, hkv, bt, d))
    q = randn_bf16(rng, (B, hq, d))
    return q, kc, vc, tables


def _check(out, ref, rows):
    g = out.float().cpu().numpy().astype(np.float64)[rows]
    d = np.abs(g - ref[rows])
    assert np.isfinite(g).all() and d.max() <= MAX_ABS and d.mean() <= MEAN_ABS, (d.max(), d.mean())


@pytest.mark.parametrize("bt", [8, 16, 32, 64])
def test_large_batch_one_merge_slot(pkv, bt):
    rng = np.random.default_rng(40 + bt)
    B, hq, hkv = 3000, 16, 2
    ctx = rng.integers(1, 70, size=B).astype(np.int32)
    ctx[::97] = 0
    q, kc, vc, tables = _batch(rng, ctx, bt, hq, hkv)
    dev = torch.device("cuda")
    t = lambda bits: pkv.bf16_from_bits(bits).to(dev)
    ws = pkv.AttentionWorkspace(B, hkv)
    scale = 128 ** -0.5
    rows = sorted(set(range(0, B, 13)) | set(range(0, B, 97)) | {B - 1})
    ref = pa.paged_decode_attention(q, kc, vc, tables, ctx, scale, seqs=rows)
    for n in (0, 57):
        out = pkv.attn_decode(t(q), t(kc), t(vc), torch.from_numpy(tables).to(dev),
                              torch.from_numpy(ctx).to(dev), scale, workspace=ws, num_ctas=n)
        torch.cuda.synchronize()
        assert ws.read_error() == 0
        assert not out[::97].any()  # empty contexts give zero rows
        _check(out, ref, rows)
    # two CTAs per SM at this size too (one merge slot instead of two)
    assert pkv.default_ctas(B) == pkv.default_ctas(64)


def test_large_batch_cascade(pkv):
    rng = np.random.default_rng(7)
    B, hq, hkv, bt = 2400, 16, 2, 16
    groups = [(list(range(8 * i, 8 * i + 8)), 3) for i in range(B // 8)]  # eight sharers of 48 tokens each
    ctx = (48 + rng.integers(1, 21, size=B)).astype(np.int32)
    q, kc, vc, tables = _batch(rng, ctx, bt, hq, hkv, shared=groups)
    dev = torch.device("cuda")
    t = lambda bits: pkv.bf16_from_bits(bits).to(dev)
    scale = 128 ** -0.5
    rows = sorted(set(range(0, B, 17)) | {B - 1})
    ref = pa.paged_decode_attention(q, kc, vc, tables, ctx, scale, seqs=rows)
    cas = pkv.Cascade(B, hq, hkv, groups)
    out = cas.decode(t(q), t(kc), t(vc), torch.from_numpy(tables).to(dev), torch.from_numpy(ctx).to(dev), scale)
    torch.cuda.synchronize()
    assert cas.read_error() == 0
    _check(out, ref, rows)
