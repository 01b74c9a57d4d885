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
    rec = {"kernel_sha256_16": bench.kernel_hash(), "workload": "llama3_8b_b64", "context_tokens": 1000,
           "dram_bytes_per_launch": 5.0e8}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.recorded_traffic("llama3_8b_b64", 1234) == 5.0e8
    assert bench.recorded_traffic("other", 2000) == 1.0e9  # scaled by context tokens
    rec["kernel_sha256_16"] = "0" * 16  # captured from other device code
    path.write_text(json.dumps(rec))
    assert bench.recorded_traffic("llama3_8b_b64", 1234) is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "absent.json"))
    assert bench.recorded_traffic("llama3_8b_b64", 1234) is None


def test_kernel_hash_covers_the_device_sources_only():
    names = sorted(os.path.basename(p) for p in bench.KERNEL_SOURCES)
    assert names == ["pkv_decode_kernel.cuh", "pkv_ptx.cuh"]
    h = bench.kernel_hash()
    assert len(h) == 16 and int(h, 16) >= 0
