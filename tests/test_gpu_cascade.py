"""Cascade attention (shared prefix blocks read once for all their sharers)
against the oracle's paged decode attention: max |err| 2e-2, mean |err|
2e-3, as for the plain kernel. Groups come from the batch's block tables
(shared_prefix_groups) or are built by hand to reach the kernels' edge cases:
several 32-row chunks per group, several 64-tile chunks per shared prefix,
sharers without private tokens, ungrouped sequences alongside."""
import numpy as np
import pytest
import torch

from oracle import paged_attention as pa, scenario
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


def _close(out, ref):
    g = out.float().cpu().numpy().astype(np.float64)
    d = np.abs(g - ref)
    assert np.isfinite(g).all() and d.max() <= MAX_ABS and d.mean() <= MEAN_ABS, (d.max(), d.mean())


@pytest.mark.parametrize("name", ["fanout", "prefix_admission"])
def test_workload_groups_from_tables(pkv, name):
    w = make_workload(name)
    ref = scenario.replay(w)
    eng = pkv.PagedKVEngine(w.pool_blocks, w.num_q_heads, w.num_kv_heads, w.head_dim, free_order=w.free_order)
    eng.load_workload_pool(w)
    eng.replay_events(w, with_content=True)
    q, k, v = w.step_inputs()
    sb = eng.prepare_step(w.batch, q, k, v, width=ref["tables"].shape[1])
    plain = eng.run_step(sb, w.scale).clone()  # copies, append, plain attention
    groups = pkv.shared_prefix_groups(sb.tables.cpu().numpy(), sb.ctx.cpu().numpy())
    assert groups and all(len(m) >= 2 and sh >= 1 for m, sh in groups)
    cas = pkv.Cascade(len(w.batch), w.num_q_heads, w.num_kv_heads, groups)
    out = cas.decode(sb.q, eng.k_cache, eng.v_cache, sb.tables, sb.ctx, w.scale)
    torch.cuda.synchronize()
    assert cas.read_error() == 0 and eng.read_errors(sb) == 0
    _close(out, ref["out"])
    assert (out.float() - plain.float()).abs().max().item() <= 2 * MAX_ABS
    out2 = cas.decode(sb.q, eng.k_cache, eng.v_cache, sb.tables, sb.ctx, w.scale)  # repeatable
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


@pytest.mark.parametrize("hq,hkv", [(64, 8), (8, 8), (32, 8)])
def test_handmade_groups_edge_cases(pkv, hq, hkv):
    rng = np.random.default_rng(hq * 100 + hkv)
    d, b = 128, 16
    shared = 150  # three 64-tile chunks
    n_members = 40 if hq == hkv else 9  # G = 1: two 32-row chunks; G = 8: three
    private = [0, 0] + rng.integers(1, 60, size=n_members - 2).tolist()  # two sharers with no private token
    lone = [5, 300, 1]  # ungrouped sequences
    ctx = [shared * b + p for p in private] + lone
    need = shared + sum(-(-p // b) for p in private) + sum(-(-c // b) for c in lone)
    nb = need + 7
    perm = rng.permutation(nb)
    width = max(-(-c // b) for c in ctx)
    tables = np.full((len(ctx), width), -1, np.int32)
    nxt = shared
    for i, c in enumerate(ctx):
        if i < n_members:
            tables[i, :shared] = perm[:shared]
            start = shared
        else:
            start = 0
        for j in range(start, -(-c // b)):
            tables[i, j] = perm[nxt]
            nxt += 1
    kc = randn_bf16(np.random.default_rng(1), (nb, hkv, b, d))
    vc = randn_bf16(np.random.default_rng(2), (nb, hkv, b, d))
    q = randn_bf16(np.random.default_rng(3), (len(ctx), hq, d))
    scale = d ** -0.5
    ref = pa.paged_decode_attention(q, kc, vc, tables, np.array(ctx), scale)
    dev = torch.device("cuda")
    t = lambda bits: pkv.bf16_from_bits(bits).to(dev)
    members = list(range(n_members))
    rng.shuffle(members)  # member order within a group is free
    cas = pkv.Cascade(len(ctx), hq, hkv, [(members, shared)])
    out = cas.decode(t(q), t(kc), t(vc), torch.from_numpy(tables).to(dev),
                     torch.tensor(ctx, dtype=torch.int32, device=dev), scale)
    torch.cuda.synchronize()
    assert cas.read_error() == 0
    _close(out, ref)


def test_plan_rejects_bad_groups(pkv):
    with pytest.raises(pkv.PkvError):
        pkv.Cascade(4, 32, 8, [([0, 1], 2), ([1, 2], 2)])  # a sequence in two groups
    with pytest.raises(pkv.PkvError):
        pkv.Cascade(4, 32, 8, [([0, 5], 2)])  # not a sequence of the batch
    with pytest.raises(pkv.PkvError):
        pkv.Cascade(4, 32, 8, [([0, 1], 0)])  # nothing shared
