"""The bounded-wait path of the decode kernel, made to run out on purpose.

Every wait of the kernel on its shared-memory rings gives up after a limit
(1 s); the CTA then raises PKV_DEVERR_TIMEOUT in the workspace's error word,
stops issuing copies, waits (bounded) for the copies it did issue and runs to
its end without further waits, so the GPU context stays usable. Here the
producer of CTA 0 is told to issue only its first few tiles
(pkv_attn_decode_wait_test): the consumer that waits on the next one gives
up. Nothing faults or hangs: the copy that never comes is one that was never
issued. After such a call the workspace is zeroed again and the next normal
call must match the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import cache_ops, paged_attention as pa
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


def _batch(rng, ctx, hq, hkv, d=128):
    ctx = np.asarray(ctx, dtype=np.int32)
    nblk = -(-ctx // 16)
    nb = int(nblk.sum()) + 2
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.full((len(ctx), int(nblk.max())), -1, np.int32)
    nxt = 0
    for s in range(len(ctx)):
        tables[s, :nblk[s]] = perm[nxt:nxt + nblk[s]]
        nxt += int(nblk[s])
    return (randn_bf16(rng, (len(ctx), hq, d)), randn_bf16(rng, (nb, hkv, 16, d)),
            randn_bf16(rng, (nb, hkv, 16, d)), tables, ctx)


@pytest.mark.parametrize("stop_tiles", [0, 5, 13])
def test_wait_runs_out_and_the_next_call_is_exact(pkv, stop_tiles):
    from paged_kv_cache_49_gb300 import _native as nat

    rng = np.random.default_rng(30 + stop_tiles)
    hq, hkv, d = 32, 8, 128
    q, kp, vp, tables, ctx = _batch(rng, [600, 300, 45], hq, hkv)
    scale = d ** -0.5
    ref = pa.paged_decode_attention(q, kp, vp, tables, ctx, scale)
    dev = torch.device("cuda")
    t = lambda bits: pkv.bf16_from_bits(bits).to(dev)
    qd, kc, vc = t(q), t(kp), t(vp)
    td, cd = torch.from_numpy(tables).to(dev), torch.from_numpy(ctx).to(dev)
    ws = pkv.AttentionWorkspace(len(ctx), hkv)
    out = torch.zeros_like(qd)
    stream = torch.cuda.current_stream().cuda_stream
    # 4 CTAs: CTA 0's range holds about 60 tiles, so the stop falls inside it
    st = nat.lib.pkv_attn_decode_wait_test(
        qd.data_ptr(), kc.data_ptr(), vc.data_ptr(), td.data_ptr(), tables.shape[1], cd.data_ptr(), len(ctx),
        hq, hkv, d, kp.shape[0], ctypes.c_float(scale), 4, ws.ptr, ws.nbytes, out.data_ptr(), stop_tiles,
        stream)
    assert st == nat.PKV_OK
    torch.cuda.synchronize()  # returns: the wait gave up instead of hanging
    err = ws.read_error(clear=False)
    assert err & pkv.DEVERR_TIMEOUT, f"error word {err:#x}"
    assert err & ~pkv.DEVERR_TIMEOUT == 0

    # a negative stop is an argument error, refused before any launch
    bad = nat.lib.pkv_attn_decode_wait_test(
        qd.data_ptr(), kc.data_ptr(), vc.data_ptr(), td.data_ptr(), tables.shape[1], cd.data_ptr(), len(ctx),
        hq, hkv, d, kp.shape[0], ctypes.c_float(scale), 4, ws.ptr, ws.nbytes, out.data_ptr(), -1, stream)
    assert bad == nat.PKV_EINVAL

    # the context is still usable: re-zero the workspace, then a normal call
    # (same grid, and the default grid) matches the oracle
    nat.lib.pkv_attn_workspace_init(ws.ptr, ws.nbytes, stream)
    for n in (4, 0):
        out = torch.full_like(qd, float("nan"))
        pkv.attn_decode(qd, kc, vc, td, cd, scale, out, workspace=ws, num_ctas=n)
        torch.cuda.synchronize()
        assert ws.read_error() == 0
        g = out.float().cpu().numpy().astype(np.float64)
        dd = np.abs(g - ref)
        assert np.isfinite(g).all() and dd.max() <= MAX_ABS and dd.mean() <= MEAN_ABS

    # and so do the other kernels: an append lands bit-exactly
    err_word = pkv.new_error_word()
    kn, vn = randn_bf16(rng, (2, hkv, d)), randn_bf16(rng, (2, hkv, d))
    slots = np.array([int(tables[0, 1]) * 16 + 3, int(tables[2, 0]) * 16 + 15], dtype=np.int64)
    pkv.append(t(kn), t(vn), torch.from_numpy(slots).to(dev), kc, vc, err_word)
    k_ref, v_ref = kp.copy(), vp.copy()
    cache_ops.append_kv(k_ref, v_ref, kn, vn, slots)
    assert pkv.read_device_error(err_word) == 0
    assert np.array_equal(pkv.bits_from_bf16(kc), k_ref) and np.array_equal(pkv.bits_from_bf16(vc), v_ref)
