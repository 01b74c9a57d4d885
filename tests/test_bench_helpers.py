"""bench.py's host-side measurement arithmetic, on the CPU: the algorithmic
bytes of a launch (the metric's byte count), the unique KV bytes of shared
blocks, and when a committed ncu traffic record applies."""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_algorithmic_bytes_count_every_term_once():
    ctx = np.array([1, 16, 17, 203])
    hq, hkv, d = 32, 8, 128
    kv = int(ctx.sum()) * hkv * d * 2 * 2
    qo = 2 * len(ctx) * hq * d * 2
    tables = (1 + 1 + 2 + 13) * 4
    assert bench.algorithmic_bytes(ctx, hq, hkv, d) == kv + qo + tables + len(ctx) * 4
    # 8-token blocks: more table entries, same K/V, q and out bytes
    assert bench.algorithmic_bytes(ctx, hq, hkv, d, block_tokens=8) - bench.algorithmic_bytes(ctx, hq, hkv, d) == \
        ((1 + 2 + 3 + 26) - (1 + 1 + 2 + 13)) * 4


def test_unique_kv_bytes_count_shared_blocks_once():
    tables = np.array([[5, 6, 7], [5, 6, 9], [1, -1, -1]])
    ctx = np.array([40, 33, 3])  # 3, 3 and 1 blocks: {5, 6, 7, 9, 1}
    assert bench.unique_kv_bytes(tables, ctx, hkv=8) == 5 * 8 * 16 * 128 * 2 * 2


def test_recorded_traffic_applies_only_to_the_profiled_kernel(tmp_path, monkeypatch):
    rec = {"kernel_sha256_16": bench.kernel_hash(),
           "records": {"llama3_8b_b64": {"context_tokens": 1000, "dram_bytes_per_launch": 5.0e8}}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.recorded_traffic("llama3_8b_b64", 1234) == (5.0e8, "measured")
    assert bench.recorded_traffic("other", 2000) == (1.0e9, "scaled from llama3_8b_b64")  # by context tokens
    rec["records"]["other"] = {"context_tokens": 3000, "dram_bytes_per_launch": 7.0e8}
    path.write_text(json.dumps(rec))
    assert bench.recorded_traffic("other", 2000) == (7.0e8, "measured")  # its own capture wins
    rec["kernel_sha256_16"] = "0" * 16  # captured from other device code
    path.write_text(json.dumps(rec))
    assert bench.recorded_traffic("llama3_8b_b64", 1234)[0] is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "absent.json"))
    assert bench.recorded_traffic("llama3_8b_b64", 1234)[0] is None


def test_kernel_hash_covers_the_device_sources_only():
    names = sorted(os.path.basename(p) for p in bench.KERNEL_SOURCES)
    assert names == ["pkv_decode_kernel.cuh", "pkv_ptx.cuh"]
    h = bench.kernel_hash()
    assert len(h) == 16 and int(h, 16) >= 0


def test_oracle_sample_and_row_split():
    ctx = np.array([131072, 5, 131072, 900, 17, 4000, 131072, 33, 131072, 131072, 60])
    rows = bench.oracle_sample(ctx)
    assert rows == sorted(set(rows))
    assert {0, 2, 6, 8} <= set(rows)  # the first four rows at the maximum
    order = np.argsort(ctx, kind="stable")
    assert set(order[::4].tolist()) <= set(rows)
    shares = bench.split_rows(rows, ctx, 3)
    assert sorted(r for sh in shares for r in sh) == rows  # every row exactly once
    assert len(shares) == 3
    assert len(bench.split_rows([1, 4], ctx, 8)) == 2  # no empty shares


def test_oracle_cores_equal_the_single_process_oracle():
    """The all-core baseline runs the committed oracle unchanged: its outputs
    over the sample equal the oracle's own replay, row for row."""
    from oracle import scenario
    from workloads import make_workload

    for name in ("tiny", "tiny_nan"):
        w = make_workload(name)
        ctx = bench.oracle_batch_ctx(w)
        ref = scenario.replay(w)
        assert np.array_equal(ctx, ref["ctx"])
        rows = bench.oracle_sample(ctx)
        pool = bench.OracleCores(name, 0, rows, ctx, 2)
        try:
            wall, busy, out = pool.step(want_out=True)
            assert wall > 0 and busy > 0 and pool.workers == 2
            for r in rows:
                assert np.array_equal(out[r], ref["out"][r])
            wall2, _, out2 = pool.step(want_out=True)  # a step is repeatable
            assert all(np.array_equal(out2[r], out[r]) for r in rows)
        finally:
            pool.close()


def test_tail_waste_counts_the_empty_slots_of_last_blocks():
    # 1 -> 15 empty slots, 16 -> 0, 17 -> 15, 203 -> 5, 0 -> no block
    assert bench.tail_waste_tokens([1, 16, 17, 203, 0]) == 15 + 0 + 15 + 5
    assert bench.tail_waste_tokens([8, 9], block_tokens=8) == 0 + 7
