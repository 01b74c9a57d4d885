"""Host side of cascade attention: the shared-prefix groups derived from a
batch's block tables (against brute force), the bytes they save, and the
plan's size functions (no GPU needed)."""
import ctypes
import random

import numpy as np
import pytest


@pytest.fixture(scope="module")
def pkv():
    from tests.conftest import build_native
    build_native()
    import paged_kv_cache_49_gb300 as m
    return m


def _brute_groups(tables, ctx, b=16):
    out = {}
    for s in range(len(ctx)):
        if ctx[s] >= b:
            out.setdefault(int(tables[s][0]), []).append(s)
    res = []
    for members in out.values():
        if len(members) < 2:
            continue
        limit = min(int(ctx[m]) // b for m in members)
        k = 0
        while k < limit and all(tables[m][k] == tables[members[0]][k] for m in members):
            k += 1
        if k:
            res.append((members, k))
    return sorted(res)


@pytest.mark.parametrize("seed", range(8))
def test_groups_match_brute_force(pkv, seed):
    rnd = random.Random(seed)
    B, W = rnd.randint(2, 30), 40
    tables = np.full((B, W), -1, np.int32)
    ctx = np.zeros(B, np.int64)
    nxt = 1000
    prefixes = [[rnd.randrange(1000) for _ in range(rnd.randint(1, 12))] for _ in range(4)]
    for s in range(B):
        pre = rnd.choice(prefixes + [[]])
        n = rnd.randint(0, W * 16)
        blocks = (n + 15) // 16
        row = (pre + [nxt + i for i in range(W)])[:blocks]
        nxt += W
        tables[s, :len(row)] = row
        ctx[s] = n
    got = sorted((sorted(m), sh) for m, sh in pkv.shared_prefix_groups(tables, ctx))
    assert got == _brute_groups(tables, ctx)


def test_saved_bytes_of_the_fanout_workload(pkv):
    from oracle import scenario
    from workloads import make_workload
    w = make_workload("fanout")
    ref = scenario.replay(w, attend=False)
    groups = pkv.shared_prefix_groups(ref["tables"], ref["ctx"])
    assert len(groups) == 16 and all(len(m) == 8 for m, _ in groups)
    # each prompt's complete blocks, shared by its 8 samples (the partial one was copied on write)
    plen = sorted(int(ref["ctx"][m[0]]) for m, _ in groups)
    assert all(sh >= 32 for _, sh in groups)
    per_block = 8 * 16 * 128 * 2 * 2
    assert pkv.cascade_saved_bytes(groups, 8) == sum(7 * sh * per_block for _, sh in groups)
    assert pkv.cascade_saved_bytes(groups, 8) > pkv.CASCADE_MIN_SAVED_BYTES
    del plen


def test_plan_argument_checks_need_no_gpu(pkv):
    """Invalid groups are refused before any device query (the sizes
    themselves depend on the device's SM count)."""
    lib = pkv._native.lib
    offs = (ctypes.c_int32 * 3)(0, 8, 12)
    shared = (ctypes.c_int32 * 2)(100, 3)
    bad = (ctypes.c_int32 * 3)(0, 8, 8)  # an empty group
    assert lib.pkv_attn_cascade_workspace_size(16, 32, 8, 2, bad, shared) == 0
    assert lib.pkv_cascade_staging_size(16, 32, 8, 2, bad, shared) == 0
    assert lib.pkv_attn_cascade_workspace_size(4, 32, 8, 2, offs, shared) == 0  # more sharers than sequences
    none = (ctypes.c_int32 * 2)(100, 0)  # nothing shared
    assert lib.pkv_attn_cascade_workspace_size(16, 32, 8, 2, offs, none) == 0
    assert lib.pkv_attn_cascade_workspace_size(16, 30, 8, 2, offs, shared) == 0  # 30 q heads over 8 kv heads
