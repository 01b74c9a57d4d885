"""The allocation-free attention entry point (pkv_attn_decode_static).

It serves callers that cannot allocate device memory (a plugin whose host
program owns every allocation, a loop that must never call cudaMalloc): its
scratch is a static device array inside the library. Called twice in a row
through the C ABI, it must agree with pkv_attn_decode (caller workspace)
within the attention tolerance of the parity tests. This file is collected
last, and also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from workloads import make_workload

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3


def test_static_scratch_entry_point_matches_workspace_entry_point():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tests.conftest import build_native
    build_native()
    import paged_kv_cache_49_gb300 as pkv
    from paged_kv_cache_49_gb300 import _native as nat

    w = make_workload("llama3_8b_b64")
    eng = pkv.PagedKVEngine(w.pool_blocks, w.num_q_heads, w.num_kv_heads, w.head_dim,
                            free_order=w.free_order)
    eng.load_workload_pool(w)
    eng.replay_events(w)
    q, k, v = w.step_inputs()
    sb = eng.prepare_step(w.batch, q, k, v)
    ref = eng.run_step(sb, w.scale).clone()  # existing entry point, caller workspace
    torch.cuda.synchronize()
    assert eng.read_errors(sb) == 0

    err = pkv.new_error_word()
    stream = torch.cuda.current_stream().cuda_stream
    B, hq, d = sb.q.shape
    nb, hkv = eng.k_cache.shape[:2]
    for _ in range(2):
        out = torch.full_like(sb.q, float("nan"))
        status = nat.lib.pkv_attn_decode_static(
            sb.q.data_ptr(), eng.k_cache.data_ptr(), eng.v_cache.data_ptr(), sb.tables.data_ptr(),
            sb.tables.shape[1], sb.ctx.data_ptr(), B, hq, hkv, d, nb, ctypes.c_float(w.scale),
            err.data_ptr(), out.data_ptr(), stream)
        assert status == nat.PKV_OK
        torch.cuda.synchronize()
        assert pkv.read_device_error(err) == 0
        diff = (out.float() - ref.float()).abs()
        assert torch.isfinite(out.float()).all()
        assert diff.max().item() <= MAX_ABS and diff.mean().item() <= MEAN_ABS

    # batches past the kernel's limit are refused before any launch
    too_many = nat.lib.pkv_attn_decode_static(
        sb.q.data_ptr(), eng.k_cache.data_ptr(), eng.v_cache.data_ptr(), sb.tables.data_ptr(),
        sb.tables.shape[1], sb.ctx.data_ptr(), nat.MAX_SEQS + 1, hq, hkv, d, nb, ctypes.c_float(w.scale),
        None, out.data_ptr(), stream)
    assert too_many == nat.PKV_EUNSUPPORTED


def test_static_scratch_entry_point_at_a_large_batch():
    """3,000 sequences: the one-merge-slot launch, through the static scratch
    and through a caller workspace."""
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tests.conftest import build_native
    build_native()
    import paged_kv_cache_49_gb300 as pkv
    from paged_kv_cache_49_gb300 import _native as nat
    from workloads import randn_bf16

    rng = np.random.default_rng(3)
    B, hq, hkv, d, bt = 3000, 16, 2, 128, 16
    ctx = rng.integers(1, 90, size=B).astype(np.int32)
    nblk = -(-ctx // bt)
    width = int(nblk.max())
    nb = int(nblk.sum()) + 4
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.full((B, width), -1, np.int32)
    nxt = 0
    for s in range(B):
        tables[s, :nblk[s]] = perm[nxt:nxt + nblk[s]]
        nxt += int(nblk[s])
    dev = torch.device("cuda")
    t = lambda bits: pkv.bf16_from_bits(bits).to(dev)
    kc, vc = t(randn_bf16(rng, (nb, hkv, bt, d))), t(randn_bf16(rng, (nb, hkv, bt, d)))
    q = t(randn_bf16(rng, (B, hq, d)))
    td, cd = torch.from_numpy(tables).to(dev), torch.from_numpy(ctx).to(dev)
    scale = d ** -0.5
    ref = pkv.attn_decode(q, kc, vc, td, cd, scale)
    err = pkv.new_error_word()
    out = torch.full_like(q, float("nan"))
    status = nat.lib.pkv_attn_decode_static(
        q.data_ptr(), kc.data_ptr(), vc.data_ptr(), td.data_ptr(), width, cd.data_ptr(), B, hq, hkv, d, nb,
        ctypes.c_float(scale), err.data_ptr(), out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert status == nat.PKV_OK
    torch.cuda.synchronize()
    assert pkv.read_device_error(err) == 0
    diff = (out.float() - ref.float()).abs()
    assert torch.isfinite(out.float()).all()
    assert diff.max().item() <= MAX_ABS and diff.mean().item() <= MEAN_ABS
