"""Block sizes other than 16 (cs2680 Lecture 10, §10.3: the block size is a
tunable that trades tail waste and table length against the kernel's
contiguous runs): append, copy and attention through the _ex entry points
against the oracle on caches of 8-, 32- and 64-token blocks."""
import numpy as np
import pytest
import torch

from oracle import cache_ops, scenario
from workloads import make_workload, randn_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tests.conftest import build_native
    build_native()
    import paged_kv_cache_49_gb300 as m
    return m


@pytest.mark.parametrize("bt", [8, 32, 64])
@pytest.mark.parametrize("name", ["tiny", "llama3_8b_b64"])
def test_attention_and_append(pkv, name, bt):
    w = make_workload(name, block_tokens=bt)
    ref = scenario.replay(w)
    eng = pkv.PagedKVEngine(w.pool_blocks, w.num_q_heads, w.num_kv_heads, w.head_dim,
                            free_order=w.free_order, block_tokens=bt)
    eng.load_workload_pool(w)
    eng.replay_events(w)
    q, k, v = w.step_inputs()
    sb = eng.prepare_step(w.batch, q, k, v, width=ref["tables"].shape[1])
    assert sb.slots.cpu().tolist() == list(ref["slots"])
    assert np.array_equal(sb.tables.cpu().numpy(), ref["tables"])
    for n in (0, 1, 7):
        out = eng.run_step(sb, w.scale, num_ctas=n)
        torch.cuda.synchronize()
        assert eng.read_errors(sb) == 0
        g = out.float().cpu().numpy().astype(np.float64)
        d = np.abs(g - ref["out"])
        assert np.isfinite(g).all() and d.max() <= 2e-2 and d.mean() <= 2e-3, (n, d.max(), d.mean())
    assert np.array_equal(pkv.bits_from_bf16(eng.k_cache), ref["k_pool"])
    assert np.array_equal(pkv.bits_from_bf16(eng.v_cache), ref["v_pool"])


@pytest.mark.parametrize("bt", [8, 32, 64])
def test_block_copy(pkv, bt):
    rng = np.random.default_rng(bt)
    NB, Hkv, D = 12, 8, 128
    kp, vp = randn_bf16(rng, (NB, Hkv, bt, D)), randn_bf16(rng, (NB, Hkv, bt, D))
    kc, vc = pkv.bf16_from_bits(kp).cuda(), pkv.bf16_from_bits(vp).cuda()
    pairs = np.array([[2, 9], [5, 0], [11, 3]], dtype=np.int32)
    pkv.block_copy(kc, vc, torch.from_numpy(pairs).cuda())
    cache_ops.copy_blocks(kp, vp, pairs)
    torch.cuda.synchronize()
    assert np.array_equal(pkv.bits_from_bf16(kc), kp) and np.array_equal(pkv.bits_from_bf16(vc), vp)
