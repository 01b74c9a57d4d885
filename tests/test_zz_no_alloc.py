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

    # sizes past the static limit are refused before any launch
    too_many = nat.lib.pkv_attn_decode_static(
        sb.q.data_ptr(), eng.k_cache.data_ptr(), eng.v_cache.data_ptr(), sb.tables.data_ptr(),
        sb.tables.shape[1], sb.ctx.data_ptr(), 4096, hq, hkv, d, nb, ctypes.c_float(w.scale),
        None, out.data_ptr(), stream)
    assert too_many == nat.PKV_ERANGE
