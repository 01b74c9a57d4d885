"""Parity of the CUDA path (through the C ABI) with the oracle.

Append, block copy and block bookkeeping must match bit for bit; attention
outputs (bf16) must be within max |err| 2e-2 and mean |err| 2e-3 of the
oracle's float64 result. Every input comes from the seeded workloads; the
oracle side replays them with its own code.
"""
import numpy as np
import pytest
import torch

from oracle import cache_ops, paged_attention as pa, scenario
from workloads import make_workload, randn_bf16

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3


@pytest.fixture(scope="module")
def pkv():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tests.conftest import build_native
    build_native()
    import paged_kv_cache_49_gb300 as m
    return m


def _close(gpu_out, ref, rows=None):
    g = gpu_out.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        g = g[rows]
    assert np.isfinite(g).all()
    d = np.abs(g - ref)
    assert d.max() <= MAX_ABS, f"max abs err {d.max()}"
    assert d.mean() <= MEAN_ABS, f"mean abs err {d.mean()}"
    return d.max(), d.mean()


def _engine_for(pkv, w, with_content=True):
    eng = pkv.PagedKVEngine(w.pool_blocks, w.num_q_heads, w.num_kv_heads, w.head_dim,
                            free_order=w.free_order)
    eng.load_workload_pool(w)
    hist = eng.replay_events(w, with_content=with_content)
    return eng, hist


def _run_workload(pkv, w, num_ctas_list=(0,)):
    ref = scenario.replay(w)
    eng, hist = _engine_for(pkv, w)
    # block manager decisions are bit-exact
    assert [(b, s, p) for b, s, p in hist] == [(b, s, [tuple(x) for x in p]) for b, s, p in ref["history"]]
    q, k, v = w.step_inputs()
    sb = eng.prepare_step(w.batch, q, k, v, width=ref["tables"].shape[1])
    assert sb.slots.cpu().tolist() == list(ref["slots"])
    assert [tuple(x) for x in sb.pairs.cpu().tolist()] == [tuple(p) for p in ref["pairs"]]
    assert np.array_equal(sb.tables.cpu().numpy(), ref["tables"])
    assert np.array_equal(sb.ctx.cpu().numpy(), ref["ctx"])
    results = {}
    for n in num_ctas_list:
        out = eng.run_step(sb, w.scale, num_ctas=n)
        torch.cuda.synchronize()
        assert eng.read_errors(sb) == 0
        results[n] = _close(out, ref["out"])
        fused = out.clone()
        sep = eng.run_step_separate(sb, w.scale, num_ctas=n)
        torch.cuda.synchronize()
        assert torch.equal(fused, sep)
    # the pools after the step (copies, appends, history) are bit-exact
    assert np.array_equal(pkv.bits_from_bf16(eng.k_cache), ref["k_pool"])
    assert np.array_equal(pkv.bits_from_bf16(eng.v_cache), ref["v_pool"])
    return eng, sb, ref, results


@pytest.mark.parametrize("name", ["tiny", "tiny_nan", "prefix_admission"])
def test_small_workloads_all_splits(pkv, name):
    w = make_workload(name)
    _run_workload(pkv, w, num_ctas_list=(0, 1, 2, 3, 7, 37, 151))


@pytest.mark.parametrize("name", ["heads_8_8", "heads_16_8", "heads_8_1", "heads_64_8"])
def test_gqa_group_sizes(pkv, name):
    """G = 1 (MHA), 2, 8 with a single KV head (MQA) and 8 with eight."""
    w = make_workload(name)
    _run_workload(pkv, w, num_ctas_list=(0, 1, 5, 40))


def test_long_single_sequence_merges_across_every_cta(pkv):
    """One 131,072-token sequence: each KV head's run is cut among ~38 CTAs,
    so its pieces merge in two levels (groups of eight, then the groups);
    the grid sizes give 1-2, 8-9, 9-10, 16-17, 17-18 and 38-39 pieces per
    pair (a lone last piece forms its own group)."""
    w = make_workload("long_single")
    _run_workload(pkv, w, num_ctas_list=(0, 7, 64, 72, 128, 136))


def test_many_short_sequences_at_the_batch_limit(pkv):
    """4,096 sequences of 1..40 tokens: thousands of short pieces per launch."""
    w = make_workload("many_short")
    _run_workload(pkv, w, num_ctas_list=(0, 33))


def test_llama3_8b_batch64(pkv):
    w = make_workload("llama3_8b_b64")
    _run_workload(pkv, w, num_ctas_list=(0, 1, 64))


def test_fanout_with_copy_on_write(pkv):
    w = make_workload("fanout")
    eng, sb, ref, _ = _run_workload(pkv, w, num_ctas_list=(0,))
    copies = sum(len(p) for _, _, p in ref["history"]) + len(ref["pairs"])
    assert copies > 0 and eng.bm.stats()["cow_copies"] == copies


def test_llama33_70b_full_size_sampled(pkv):
    """Full-size 256-sequence, 64/8-head batch with four 131,072-token
    contexts, in the bench's launch configuration; the oracle computes the
    four long rows and a seeded sample of the rest."""
    w = make_workload("llama33_70b_b256")
    eng, _ = _engine_for(pkv, w, with_content=False)
    q, k, v = w.step_inputs()
    sb = eng.prepare_step(w.batch, q, k, v)
    out = eng.run_step(sb, w.scale)
    torch.cuda.synchronize()
    assert eng.read_errors(sb) == 0
    rng = np.random.default_rng(123)
    rows = [0, 1, 2, 3] + sorted(rng.choice(np.arange(4, 256), size=12, replace=False).tolist())
    ref_rows, book = scenario.replay_sampled(w, rows)
    assert sb.slots.cpu().tolist() == list(book["slots"])
    assert np.array_equal(sb.ctx.cpu().numpy(), book["ctx"])
    _close(out, ref_rows, rows)


def test_unsplit_identical_rows_are_bit_identical(pkv):
    # cs2680 §10.4: shared blocks hold identical K/V, so identical queries
    # over identical tables give identical outputs.
    w = make_workload("tiny")
    eng, _ = _engine_for(pkv, w)
    q, k, v = w.step_inputs()
    sb = eng.prepare_step(w.batch, q, k, v)
    eng.run_step(sb, w.scale)
    tables = torch.cat([sb.tables[3:4], sb.tables[3:4]])
    ctx = torch.cat([sb.ctx[3:4], sb.ctx[3:4]])
    qq = torch.cat([sb.q[3:4], sb.q[3:4]])
    out = pkv.attn_decode(qq, eng.k_cache, eng.v_cache, tables, ctx, w.scale, num_ctas=1)
    assert torch.equal(out[0], out[1])
    out = pkv.attn_decode(qq, eng.k_cache, eng.v_cache, tables, ctx, w.scale)
    assert (out[0].float() - out[1].float()).abs().max().item() <= MAX_ABS


def test_workspace_reuse_and_repeat(pkv):
    w = make_workload("llama3_8b_b64")
    eng, _ = _engine_for(pkv, w)
    q, k, v = w.step_inputs()
    sb = eng.prepare_step(w.batch, q, k, v)
    a = eng.run_step(sb, w.scale).clone()
    for _ in range(3):
        b = eng.run_step(sb, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert (sb.workspace.tensor[256: 256 + 4 * 64 * 8].view(torch.int32) == 0).all()


def test_zero_and_clamped_contexts_and_bad_ids(pkv):
    rng = np.random.default_rng(5)
    NB, Hq, Hkv, D = 32, 32, 8, 128
    kp, vp = randn_bf16(rng, (NB, Hkv, 16, D)), randn_bf16(rng, (NB, Hkv, 16, D))
    q = randn_bf16(rng, (4, Hq, D))
    tables = rng.permutation(NB)[:12].reshape(4, 3).astype(np.int32)
    ctx = np.array([0, 40, 48, 33], dtype=np.int32)
    dev = "cuda"
    kc, vc = pkv.bf16_from_bits(kp).to(dev), pkv.bf16_from_bits(vp).to(dev)
    qd = pkv.bf16_from_bits(q).to(dev)
    ws = pkv.AttentionWorkspace(4, Hkv)
    out = pkv.attn_decode(qd, kc, vc, torch.from_numpy(tables).to(dev), torch.from_numpy(ctx).to(dev),
                          0.088, workspace=ws)
    ref = pa.paged_decode_attention(q, kp, vp, tables, ctx, 0.088)
    assert not out[0].any()
    _close(out, ref)
    assert ws.read_error() == 0
    # a context past the table width is clamped and flagged
    ctx2 = ctx.copy()
    ctx2[1] = 60
    out = pkv.attn_decode(qd, kc, vc, torch.from_numpy(tables).to(dev), torch.from_numpy(ctx2).to(dev),
                          0.088, workspace=ws)
    assert ws.read_error() == pkv.DEVERR_CONTEXT
    _close(out[1:2], pa.paged_decode_attention(q[1:2], kp, vp, tables[1:2], np.array([48]), 0.088))
    # an out-of-range block id never faults: it is flagged, and other rows stay right
    bad = tables.copy()
    bad[3, 2] = NB + 5
    out = pkv.attn_decode(qd, kc, vc, torch.from_numpy(bad).to(dev), torch.from_numpy(ctx).to(dev),
                          0.088, workspace=ws)
    assert ws.read_error() == pkv.DEVERR_BLOCK_ID
    _close(out[:3], ref[:3], None)


def test_many_empty_contexts_between_short_and_long(pkv):
    """Half the batch has no context, interleaved with 1..300-token and
    900-token sequences: the work partition leaves cost gaps that hold no
    tile, so some CTAs get no work and others start or end inside a gap."""
    rng = np.random.default_rng(11)
    B, Hq, Hkv, D, W = 40, 16, 2, 128, 64
    NB = 400
    kp, vp = randn_bf16(rng, (NB, Hkv, 16, D)), randn_bf16(rng, (NB, Hkv, 16, D))
    q = randn_bf16(rng, (B, Hq, D))
    tables = rng.integers(0, NB, size=(B, W)).astype(np.int32)
    ctx = np.where(np.arange(B) % 2 == 0, 0, rng.integers(1, 301, size=B)).astype(np.int32)
    ctx[[5, 17, 33]] = 900
    ref = pa.paged_decode_attention(q, kp, vp, tables, ctx, 0.088)
    dev = "cuda"
    kc, vc = pkv.bf16_from_bits(kp).to(dev), pkv.bf16_from_bits(vp).to(dev)
    qd = pkv.bf16_from_bits(q).to(dev)
    td, cd = torch.from_numpy(tables).to(dev), torch.from_numpy(ctx).to(dev)
    ws = pkv.AttentionWorkspace(B, Hkv)
    for n in (0, 1, 2, 3, 9, 64, 151, 300):
        out = pkv.attn_decode(qd, kc, vc, td, cd, 0.088, workspace=ws, num_ctas=n)
        torch.cuda.synchronize()
        assert ws.read_error() == 0
        assert not out[0::2].any()
        _close(out, ref)


def test_append_and_copy_bit_exact_with_padding_and_bad_slots(pkv):
    rng = np.random.default_rng(6)
    NB, Hkv, D = 24, 8, 128
    kp, vp = randn_bf16(rng, (NB, Hkv, 16, D)), randn_bf16(rng, (NB, Hkv, 16, D))
    kc, vc = pkv.bf16_from_bits(kp).cuda(), pkv.bf16_from_bits(vp).cuda()
    err = pkv.new_error_word()
    kn, vn = randn_bf16(rng, (6, Hkv, D)), randn_bf16(rng, (6, Hkv, D))
    slots = np.array([5, -1, 16 * 7 + 15, 16 * 23, NB * 16 + 3, 200], dtype=np.int64)
    pkv.append(pkv.bf16_from_bits(kn).cuda(), pkv.bf16_from_bits(vn).cuda(),
               torch.from_numpy(slots).cuda(), kc, vc, err)
    assert pkv.read_device_error(err) == pkv.DEVERR_SLOT
    k_ref, v_ref = kp.copy(), vp.copy()
    ok = np.where(slots < NB * 16, slots, -1)
    cache_ops.append_kv(k_ref, v_ref, kn, vn, ok)
    assert np.array_equal(pkv.bits_from_bf16(kc), k_ref) and np.array_equal(pkv.bits_from_bf16(vc), v_ref)
    pairs = np.array([[3, 9], [12, 0], [7, 20], [1, NB + 1]], dtype=np.int32)
    pkv.block_copy(kc, vc, torch.from_numpy(pairs).cuda(), err)
    assert pkv.read_device_error(err) == pkv.DEVERR_BLOCK_ID
    cache_ops.copy_blocks(k_ref, v_ref, pairs[:3])
    assert np.array_equal(pkv.bits_from_bf16(kc), k_ref) and np.array_equal(pkv.bits_from_bf16(vc), v_ref)


def test_one_workspace_serves_any_launch_shape(pkv):
    """One workspace, calls of different batches, KV-head counts and grids in
    turn, with the bytes past the counters filled with garbage before each
    call (what earlier launches leave in their partial slots): every call
    must match the oracle. Pairs of 313 tiles are cut among up to ~100 CTAs,
    so their merges run in two levels (group counters) as well as one."""
    rng = np.random.default_rng(21)
    D, dev = 128, "cuda"
    # the header (error word) and the merge counters come first;
    # nothing after them has to start at zero
    counters_end = pkv.AttentionWorkspace.fixed_bytes()
    assert counters_end % 256 == 0 and counters_end > 256
    shapes = []
    for B, Hq, Hkv, ctx in ((3, 16, 2, [5000, 37, 1200]), (40, 32, 8, None), (1, 8, 1, [20000])):
        if ctx is None:
            ctx = rng.integers(1, 700, size=B).tolist()
            ctx[7] = 4000
        ctx = np.array(ctx, dtype=np.int32)
        nblk = -(-ctx // 16)
        NB = int(nblk.sum()) + 3
        perm = rng.permutation(NB).astype(np.int32)
        tables = np.full((B, int(nblk.max())), -1, np.int32)
        nxt = 0
        for s in range(B):
            tables[s, :nblk[s]] = perm[nxt:nxt + nblk[s]]
            nxt += int(nblk[s])
        kp, vp = randn_bf16(rng, (NB, Hkv, 16, D)), randn_bf16(rng, (NB, Hkv, 16, D))
        q = randn_bf16(rng, (B, Hq, D))
        ref = pa.paged_decode_attention(q, kp, vp, tables, ctx, D ** -0.5)
        shapes.append(dict(ref=ref, q=pkv.bf16_from_bits(q).to(dev), k=pkv.bf16_from_bits(kp).to(dev),
                           v=pkv.bf16_from_bits(vp).to(dev), t=torch.from_numpy(tables).to(dev),
                           c=torch.from_numpy(ctx).to(dev)))
    ws = pkv.AttentionWorkspace(64, 8)
    for i, (which, n) in enumerate([(0, 300), (0, 64), (1, 151), (0, 9), (2, 300), (1, 0), (2, 17), (0, 0)]):
        sh = shapes[which]
        ws.tensor[counters_end:].fill_(0x5B + i)
        out = torch.full_like(sh["q"], float("nan"))
        pkv.attn_decode(sh["q"], sh["k"], sh["v"], sh["t"], sh["c"], D ** -0.5, out, workspace=ws, num_ctas=n)
        torch.cuda.synchronize()
        assert ws.read_error() == 0
        assert not ws.tensor[4:counters_end].any(), "counters left nonzero"
        _close(out, sh["ref"])


def test_default_grid_follows_the_tables_bound(pkv):
    """With num_ctas = 0 a batch whose block tables bound its work to under
    4 cost units per CTA (tiles plus 3 per sequence and KV head, every row
    full) launches fewer CTAs than fit; larger batches launch every CTA."""
    assert pkv.launch_ctas(4, 8, 13) == min(pkv.default_ctas(4), -(-8 * 4 * (13 + 3) // 4))
    assert pkv.launch_ctas(6, 1, 33) == min(pkv.default_ctas(6), -(-6 * (33 + 3) // 4))
    assert pkv.launch_ctas(64, 8, 512) == pkv.default_ctas(64)
    assert pkv.launch_ctas(8, 8, 145) == pkv.default_ctas(8)
    assert pkv.launch_ctas(4, 8, 26, 8) == pkv.launch_ctas(4, 8, 13, 16)  # the bound counts 16-token tiles
    assert pkv.launch_ctas(4, 8, 13, 12) == 0  # an unsupported block size
