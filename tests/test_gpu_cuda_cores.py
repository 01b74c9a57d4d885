"""Parity of the CUDA-core variant of the decode kernel with the oracle.

pkv_attn_decode_cuda_cores runs the same kernel with the per-tile math --
the dot products of the query heads with each key and the probability-
weighted sum of the values -- on the FP32 pipe instead of the tensor cores.
It exists to measure the tensor-core choice, so it is held to the same
attention tolerance (max |err| 2e-2, mean 2e-3 against the float64 oracle)
on the group sizes it serves: 4 (the Llama-3-8B geometry) and 8 (the
Llama-3.3-70B geometry), across grid sizes that split pairs among many CTAs.
"""
import numpy as np
import pytest
import torch

from oracle import scenario
from workloads import make_workload

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


def _step(pkv, w, with_content=True):
    eng = pkv.PagedKVEngine(w.pool_blocks, w.num_q_heads, w.num_kv_heads, w.head_dim, free_order=w.free_order)
    eng.load_workload_pool(w)
    eng.replay_events(w, with_content=with_content)
    q, k, v = w.step_inputs()
    sb = eng.prepare_step(w.batch, q, k, v)
    tensor = eng.run_step(sb, w.scale).clone()  # append, then the tensor-core attention
    torch.cuda.synchronize()
    assert eng.read_errors(sb) == 0
    return eng, sb, tensor


@pytest.mark.parametrize("name,grids", [("llama3_8b_b64", (0, 1, 64, 151)), ("tiny", (0, 1, 3, 37)),
                                        ("heads_64_8", (0, 1, 5, 40)), ("long_single", (0, 7, 72))])
def test_cuda_core_variant_matches_the_oracle(pkv, name, grids):
    w = make_workload(name)
    ref = scenario.replay(w)
    eng, sb, tensor = _step(pkv, w)
    for n in grids:
        out = torch.full_like(sb.q, float("nan"))
        pkv.attn_decode_cuda_cores(sb.q, eng.k_cache, eng.v_cache, sb.tables, sb.ctx, w.scale, out,
                                   sb.workspace, num_ctas=n)
        torch.cuda.synchronize()
        assert sb.workspace.read_error() == 0
        _close(out, ref["out"])
    # and it agrees with the tensor-core kernel within the same tolerance
    d = (out.float() - tensor.float()).abs()
    assert d.max().item() <= MAX_ABS and d.mean().item() <= MEAN_ABS


def test_cuda_core_variant_at_the_70b_size(pkv):
    """The 256-sequence Llama-3.3-70B batch (G = 8, four 131,072-token
    contexts) in the default launch; the oracle computes a sample of rows."""
    w = make_workload("llama33_70b_b256")
    eng, sb, _ = _step(pkv, w, with_content=False)
    out = pkv.attn_decode_cuda_cores(sb.q, eng.k_cache, eng.v_cache, sb.tables, sb.ctx, w.scale)
    torch.cuda.synchronize()
    rng = np.random.default_rng(321)
    rows = [0, 1, 2, 3] + sorted(rng.choice(np.arange(4, 256), size=8, replace=False).tolist())
    ref_rows, _ = scenario.replay_sampled(w, rows)
    _close(out, ref_rows, rows)


def test_cuda_core_variant_refuses_other_group_sizes(pkv):
    w = make_workload("heads_16_8")  # G = 2
    eng, sb, _ = _step(pkv, w)
    with pytest.raises(pkv.PkvError) as e:
        pkv.attn_decode_cuda_cores(sb.q, eng.k_cache, eng.v_cache, sb.tables, sb.ctx, w.scale)
    assert e.value.status == -6  # PKV_EUNSUPPORTED


@pytest.mark.parametrize("hq", [8, 16])
def test_cuda_core_variant_at_a_large_batch(pkv, hq):
    """3,000 sequences: the one-merge-slot instantiations of the variant
    (group sizes 4 and 8), empty contexts included, on a sample of rows."""
    from oracle import paged_attention as pa
    from workloads import randn_bf16

    rng = np.random.default_rng(50 + hq)
    B, hkv, d, bt = 3000, 2, 128, 16
    ctx = rng.integers(1, 90, size=B).astype(np.int32)
    ctx[::101] = 0
    nblk = -(-ctx // bt)
    width = int(nblk.max())
    nb = int(nblk.sum()) + 4
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.full((B, width), -1, np.int32)
    nxt = 0
    for s in range(B):
        tables[s, :nblk[s]] = perm[nxt:nxt + nblk[s]]
        nxt += int(nblk[s])
    kp, vp = randn_bf16(rng, (nb, hkv, bt, d)), randn_bf16(rng, (nb, hkv, bt, d))
    q = randn_bf16(rng, (B, hq, d))
    dev = torch.device("cuda")
    t = lambda bits: pkv.bf16_from_bits(bits).to(dev)
    scale = d ** -0.5
    rows = sorted(set(range(0, B, 11)) | set(range(0, B, 101)) | {B - 1})
    ref = pa.paged_decode_attention(q, kp, vp, tables, ctx, scale, seqs=rows)
    ws = pkv.AttentionWorkspace(B, hkv)
    out = torch.full((B, hq, d), float("nan"), dtype=torch.bfloat16, device=dev)
    pkv.attn_decode_cuda_cores(t(q), t(kp), t(vp), torch.from_numpy(tables).to(dev), torch.from_numpy(ctx).to(dev),
                               scale, out, ws)
    torch.cuda.synchronize()
    assert ws.read_error() == 0
    assert (out[::101] == 0).all().item()  # empty contexts give zero rows
    _close(out, ref[rows], rows)
