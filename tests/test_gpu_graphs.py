"""Decode steps replayed from CUDA graphs captured per batch bucket ("The
inference server": pad the batch to a bucket, copy tables and lengths into
the captured buffers, replay) must equal the eager library calls bit for
bit, and the eager path equals the oracle (tests/test_gpu_parity.py)."""
import numpy as np
import pytest
import torch

from oracle import scenario
from workloads import make_workload, randn_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tests.conftest import build_native
    build_native()
    import paged_kv_cache_49_gb300 as m
    return m


def _pair(pkv, w):
    engines = []
    for _ in range(2):
        e = pkv.PagedKVEngine(w.pool_blocks, w.num_q_heads, w.num_kv_heads, w.head_dim, free_order=w.free_order)
        e.load_workload_pool(w)
        e.replay_events(w)
        engines.append(e)
    return engines


@pytest.mark.parametrize("name,subsets", [
    ("llama3_8b_b64", [[5], [0, 9, 17], list(range(10, 15)), list(range(64)), [63, 1, 2, 3, 4, 5, 6]]),
    ("prefix_admission", [list(range(8)), [7], [0]]),
])
def test_graphed_steps_equal_eager_steps(pkv, name, subsets):
    w = make_workload(name)
    eager, graphed = _pair(pkv, w)
    width = max(len(eager.bm.table(s)) for s in w.batch)
    dec = pkv.GraphedDecoder(graphed, max_batch=len(w.batch), max_blocks_per_seq=width, scale=w.scale)
    rng = np.random.default_rng(7)
    saw_pairs = False
    for ids in subsets:
        q = randn_bf16(rng, (len(ids), w.num_q_heads, w.head_dim))
        k = randn_bf16(rng, (len(ids), w.num_kv_heads, w.head_dim))
        v = randn_bf16(rng, (len(ids), w.num_kv_heads, w.head_dim))
        sb = eager.prepare_step(ids, q, k, v, width=width)
        out_e = eager.run_step(sb, w.scale)
        out_g, slots, pairs = dec.step_bits(ids, q, k, v)
        torch.cuda.synchronize()
        saw_pairs |= bool(pairs)
        assert sb.slots.cpu().tolist() == slots
        assert [tuple(p) for p in sb.pairs.cpu().tolist()] == [tuple(p) for p in pairs]
        assert torch.equal(out_e, out_g), f"batch {ids}"
        assert eager.read_errors(sb) == 0 and pkv.read_device_error(graphed.error) == 0
    assert torch.equal(eager.k_cache, graphed.k_cache) and torch.equal(eager.v_cache, graphed.v_cache)
    if name == "prefix_admission":
        assert saw_pairs  # the forked request's first write copied its shared block


def test_graphed_step_matches_oracle_with_padding(pkv):
    w = make_workload("tiny")
    ref = scenario.replay(w)
    eng = pkv.PagedKVEngine(w.pool_blocks, w.num_q_heads, w.num_kv_heads, w.head_dim, free_order=w.free_order)
    eng.load_workload_pool(w)
    eng.replay_events(w)
    dec = pkv.GraphedDecoder(eng, max_batch=8, max_blocks_per_seq=ref["tables"].shape[1], scale=w.scale,
                             buckets=[8])
    q, k, v = w.step_inputs()  # 4 sequences padded to the only bucket, 8
    out, slots, _ = dec.step_bits(w.batch, q, k, v)
    torch.cuda.synchronize()
    assert slots == list(ref["slots"])
    g = out.float().cpu().numpy().astype(np.float64)
    d = np.abs(g - ref["out"])
    assert d.max() <= 2e-2 and d.mean() <= 2e-3
    assert np.array_equal(pkv.bits_from_bf16(eng.k_cache), ref["k_pool"])
