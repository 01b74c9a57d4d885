"""The oracle's replay of the synthetic workloads reproduces the accounting the
pages fix and the closed forms of the decode step."""
import numpy as np

from oracle import paged_attention as pa, scenario
from workloads import make_workload


def test_tiny_uses_seventeen_pages_and_ctx1_returns_new_value():
    w = make_workload("tiny")
    r = scenario.replay(w)
    assert r["bm"].stats()["used"] == 17
    assert list(r["ctx"]) == [1, 16, 17, 203]
    q, k_new, v_new = w.step_inputs()
    for h in range(w.num_q_heads):  # ctx 1: the output is the appended value
        assert np.array_equal(r["out"][0, h], pa.widen_bf16(v_new[0, h // 4]))


def test_prefix_admission_accounting():
    w = make_workload("prefix_admission")
    r = scenario.replay(w, attend=False)
    st = r["bm"].stats()
    # 128 shared + 7 x 17 private = 247; the fork of request 0 (ctx 2248,
    # 141 pages written, last one partial) reserves 4 pages and one spare;
    # the step's first write to the shared partial block copies it.
    assert len(r["pairs"]) == 1
    assert st["used"] == 247 + 5 and st["spares"] == 0 and st["free"] == 256 - 252
    assert r["ctx"][0] == 2249 and r["ctx"][7] == 2249


def test_fanout_copies_on_divergence():
    w = make_workload("fanout")
    r = scenario.replay(w, attend=False)
    copies = sum(len(p) for _, _, p in r["history"]) + len(r["pairs"])
    partial_prompts = sum(1 for ev in w.events if ev[0] == "admit" and ev[1] % 16)
    assert copies == 7 * partial_prompts
    assert r["bm"].stats()["spares"] == 0


def test_sampled_replay_matches_full_replay():
    w = make_workload("llama3_8b_b64")
    full = scenario.replay(w)
    rows = [0, 5, 17, 63]
    out, _ = scenario.replay_sampled(w, rows)
    assert np.array_equal(out, full["out"][rows])
