"""The host-buffer decode step (packed inputs staged from host memory, the
step, output rows back in host memory) against the device-resident step:
identical output rows and pools, bit for bit, and the oracle within
tolerance."""
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


def _engine(pkv, w):
    eng = pkv.PagedKVEngine(w.pool_blocks, w.num_q_heads, w.num_kv_heads, w.head_dim, free_order=w.free_order)
    eng.load_workload_pool(w)
    eng.replay_events(w, with_content=True)
    return eng


@pytest.mark.parametrize("name", ["tiny", "prefix_admission", "fanout"])
def test_host_step_matches_device_step(pkv, name):
    w = make_workload(name)
    ref = scenario.replay(w)
    q, k, v = w.step_inputs()
    width = ref["tables"].shape[1]
    dev = _engine(pkv, w)
    sb = dev.prepare_step(w.batch, q, k, v, width=width)
    out_dev = dev.run_step(sb, w.scale).clone()
    host = _engine(pkv, w)
    slots, pairs = host.bm.prepare_append(w.batch)
    tables, ctx = host.bm.batch_tables(w.batch, width)
    step = pkv.HostStep(host, len(w.batch), width, max_pairs=len(w.batch))
    step.pack(pkv.bf16_from_bits(q), pkv.bf16_from_bits(k), pkv.bf16_from_bits(v), slots, tables, ctx, pairs)
    out = step.run(w.scale)
    torch.cuda.synchronize()
    assert host.read_errors() == 0 and step.workspace.read_error() == 0
    assert torch.equal(out, out_dev.cpu())
    assert torch.equal(host.k_cache, dev.k_cache) and torch.equal(host.v_cache, dev.v_cache)
    d = np.abs(out.float().numpy().astype(np.float64) - ref["out"])
    assert d.max() <= MAX_ABS and d.mean() <= MEAN_ABS
    # the step is idempotent for fixed inputs: running it again from the same
    # buffers gives the same rows and pools
    step.run(w.scale)
    torch.cuda.synchronize()  # out_host is valid once the stream has passed the step
    out_again = step.out_host.clone()
    assert torch.equal(out_again, out_dev.cpu())
    assert torch.equal(host.k_cache, dev.k_cache) and torch.equal(host.v_cache, dev.v_cache)


def test_host_step_output_to_pageable_memory(pkv):
    """Pinned host_out is written by the kernel directly; pageable host_out
    goes through device_out and one copy. Both give the same rows."""
    w = make_workload("tiny")
    q, k, v = w.step_inputs()
    eng = _engine(pkv, w)
    slots, pairs = eng.bm.prepare_append(w.batch)
    width = 16
    tables, ctx = eng.bm.batch_tables(w.batch, width)
    step = pkv.HostStep(eng, len(w.batch), width, max_pairs=4)
    step.pack(pkv.bf16_from_bits(q), pkv.bf16_from_bits(k), pkv.bf16_from_bits(v), slots, tables, ctx, pairs)
    step.run(w.scale)
    torch.cuda.synchronize()
    pinned = step.out_host.clone()
    pageable = torch.empty_like(step.out_host)  # not pinned
    assert not pageable.is_pinned()
    pkv.decode_step_host(step.host, step.staging, step.num_pairs, eng.k_cache, eng.v_cache, width, len(w.batch),
                         w.num_q_heads, w.scale, step.workspace, step.out_dev, pageable, eng.error)
    torch.cuda.synchronize()
    assert torch.equal(pinned, pageable) and torch.equal(step.out_dev.cpu(), pageable)


def test_host_step_inputs_from_pageable_memory(pkv):
    """Pinned host_packed is staged by a kernel reading it across the host
    link; pageable host_packed (and a pinned buffer at an offset that is not
    16-byte aligned) go through one copy. All give the same rows and pools."""
    w = make_workload("tiny")
    q, k, v = w.step_inputs()
    outs, pools = [], []
    for mode in ("pinned", "pageable", "unaligned"):
        eng = _engine(pkv, w)
        slots, pairs = eng.bm.prepare_append(w.batch)
        width = 16
        tables, ctx = eng.bm.batch_tables(w.batch, width)
        step = pkv.HostStep(eng, len(w.batch), width, max_pairs=4)
        step.pack(pkv.bf16_from_bits(q), pkv.bf16_from_bits(k), pkv.bf16_from_bits(v), slots, tables, ctx, pairs)
        packed = step.host
        if mode == "pageable":
            packed = step.host.clone()
            assert not packed.is_pinned()
        elif mode == "unaligned":
            big = torch.empty(packed.numel() + 8, dtype=torch.uint8).pin_memory()
            big[8:].copy_(packed)
            packed = big[8:]
        pkv.decode_step_host(packed, step.staging, step.num_pairs, eng.k_cache, eng.v_cache, width, len(w.batch),
                             w.num_q_heads, w.scale, step.workspace, step.out_dev, step.out_host, eng.error)
        torch.cuda.synchronize()
        assert eng.read_errors() == 0 and step.workspace.read_error() == 0
        outs.append(step.out_host.clone())
        pools.append((eng.k_cache.clone(), eng.v_cache.clone()))
    for o, (kc, vc) in zip(outs[1:], pools[1:]):
        assert torch.equal(o, outs[0]) and torch.equal(kc, pools[0][0]) and torch.equal(vc, pools[0][1])


def test_host_step_stages_only_live_table_entries(pkv):
    """The staging kernel brings every field of the packed inputs but the
    block tables whole, and of each table row only the 16-byte words that
    hold its entries up to ceil(context_len / 16); the rest of each row in
    the device buffer keeps what it held. Rows of 13 entries (52 bytes) start
    mid-word; one row has no context."""
    w = make_workload("tiny")
    q, k, v = w.step_inputs()
    host = _engine(pkv, w)
    slots, pairs = host.bm.prepare_append(w.batch)
    width = 13
    tables, ctx = host.bm.batch_tables(w.batch, width)
    ctx[1] = 0  # a row with no context: none of its entries cross
    step = pkv.HostStep(host, len(w.batch), width, max_pairs=len(w.batch))
    step.pack(pkv.bf16_from_bits(q), pkv.bf16_from_bits(k), pkv.bf16_from_bits(v), slots, tables, ctx, pairs)
    step.staging.fill_(0xA5)
    step.run(w.scale)
    torch.cuda.synchronize()
    assert host.read_errors() == 0 and step.workspace.read_error() == 0
    dev = step.staging.cpu().numpy()
    src = step.host.numpy()
    # the layout for this step's pairs (the buffers are sized for max_pairs)
    lay = pkv.step_layout(len(w.batch), w.num_q_heads, w.num_kv_heads, w.head_dim, width, step.num_pairs)
    t0, t1, end = lay["block_tables"], lay["context_lens"], lay["bytes"]
    assert np.array_equal(dev[:t0], src[:t0]) and np.array_equal(dev[t1:end], src[t1:end])
    copied = np.zeros(t1 - t0, dtype=bool)
    for r, c in enumerate(ctx.tolist()):
        live = min(max((c + 15) // 16, 0), width)
        a = t0 + r * width * 4
        if live:
            copied[(a // 16) * 16 - t0: ((a + live * 4 + 15) // 16) * 16 - t0] = True
        assert np.array_equal(dev[a: a + live * 4], src[a: a + live * 4])
    assert (dev[t0:t1][~copied] == 0xA5).all()  # nothing else of the tables crossed
    assert step.h2d_bytes() == (lay["bytes"] - (t1 - t0)) + int(copied.sum())
