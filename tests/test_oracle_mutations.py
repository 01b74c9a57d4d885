"""The pins must catch plausible mistakes: each case plants one error in the
oracle (on the CPU, by monkeypatching) and checks that a pin test fails."""
import json
import os

import numpy as np
import pytest

import oracle.accounting as acc
import oracle.block_manager as bmod
import oracle.paged_attention as pa
from tests import test_oracle_attention as ta
from tests import test_oracle_block_manager as tb

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_numbers.json")))


def _wrong_gqa(q, k_cache, v_cache, block_tables, context_lens, scale, seqs=None):
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    out = np.zeros((B, Hq, D))
    qf = pa.widen_bf16(q)
    for s in range(B):
        n = int(context_lens[s])
        for h in range(Hq):
            g = h % Hkv  # planted: interleaved instead of grouped heads
            keys = pa.gather_tokens(k_cache, block_tables[s], n, g)
            vals = pa.gather_tokens(v_cache, block_tables[s], n, g)
            out[s, h] = pa.attend_one(qf[s, h], keys, vals, scale)
    return out


def _gather_row_off_by_one(cache, table_row, ctx, kv_head):
    b = cache.shape[2]
    t = np.arange(ctx)
    return pa.widen_bf16(cache[table_row[t // b], kv_head, (t + 1) % b, :])


def _gather_without_table(cache, table_row, ctx, kv_head):
    b = cache.shape[2]
    t = np.arange(ctx)
    return pa.widen_bf16(cache[t // b, kv_head, t % b, :])  # planted: logical block used as physical


def _attend_no_scale(q_vec, keys, values, scale):
    x = np.einsum("td,d->t", keys, q_vec)
    w = np.exp(x - x.max())
    return np.einsum("t,td->d", w, values) / w.sum()


def _attend_no_shift(q_vec, keys, values, scale):
    x = scale * np.einsum("td,d->t", keys, q_vec)
    with np.errstate(over="ignore", invalid="ignore"):
        w = np.exp(x)
        return np.einsum("t,td->d", w, values) / w.sum()


def _attend_transposed(q_vec, keys, values, scale):
    x = scale * np.einsum("td,d->t", values, q_vec)  # planted: scores against V
    w = np.exp(x - x.max())
    return np.einsum("t,td->d", w, keys) / w.sum()


def _attend_unnormalised(q_vec, keys, values, scale):
    x = scale * np.einsum("td,d->t", keys, q_vec)
    w = np.exp(x - x.max())
    return np.einsum("t,td->d", w, values)


ATTENTION_PINS = [
    lambda: ta.test_matches_sdpa_on_dense_cache(32, 8),
    ta.test_brute_force_pure_python,
    ta.test_two_token_weights_and_no_overflow,
    ta.test_equal_keys_average_the_values,
    ta.test_gqa_head_mapping,
]


def _fails(pins):
    failures = 0
    for pin in pins:
        try:
            pin()
        except (Exception, pytest.fail.Exception):  # noqa: BLE001 - any failure counts as caught
            failures += 1
    return failures


@pytest.mark.parametrize("target,replacement", [
    ("paged_decode_attention", _wrong_gqa),
    ("gather_tokens", _gather_row_off_by_one),
    ("gather_tokens", _gather_without_table),
    ("attend_one", _attend_no_scale),
    ("attend_one", _attend_no_shift),
    ("attend_one", _attend_transposed),
    ("attend_one", _attend_unnormalised),
])
def test_attention_mistake_is_caught(monkeypatch, target, replacement):
    monkeypatch.setattr(pa, target, replacement)
    assert _fails(ATTENTION_PINS) >= 1


def test_floor_pages_is_caught(monkeypatch):
    monkeypatch.setattr(acc, "request_pages", lambda p, o, b=16: (p + o) // b)
    assert _fails([lambda: tb.test_admission_arithmetic(GOLDEN)]) == 1


def test_charging_shared_pages_per_request_is_caught(monkeypatch):
    real_admit = bmod.BlockManager.admit

    def admit(self, prompt_len, max_new, group=-1, prefix_len=0):
        return real_admit(self, prompt_len, max_new, -1, 0)  # planted: no sharing

    monkeypatch.setattr(bmod.BlockManager, "admit", admit)
    assert _fails([lambda: tb.test_block_manager_shared_prefix_admission(GOLDEN)]) == 1


def test_copy_without_refcount_is_caught(monkeypatch):
    real = bmod.BlockManager.prepare_append

    def prepare_append(self, seq_ids):
        saved = list(self.ref)
        self.ref = [min(r, 1) for r in self.ref]  # planted: never sees sharing
        try:
            return real(self, seq_ids)
        finally:
            self.ref = [max(a, b) if a > 1 else b for a, b in zip(saved, self.ref)]

    monkeypatch.setattr(bmod.BlockManager, "prepare_append", prepare_append)
    assert _fails([tb.test_copy_on_write_refcount_board]) == 1


# -- incremental policy and prefix cache -----------------------------------

from tests import test_oracle_block_policies as tp  # noqa: E402


def _policy_pins():
    pins = [lambda: tp.test_prefix_hit_worked_example(GOLDEN), lambda: tp.test_two_users_share_system_prompt(GOLDEN),
            tp.test_hits_are_prefix_only, tp.test_partial_prompt_block_is_not_indexed,
            tp.test_eviction_is_lru_leaf_first_and_spares_pinned_blocks,
            tp.test_eviction_prefers_least_recently_released, tp.test_hit_on_idle_block_is_not_double_counted,
            lambda: tp.test_incremental_admits_more_than_full_reservation(GOLDEN),
            lambda: tp.test_growth_failure_then_preempt_newest_then_resume(GOLDEN),
            tp.test_watermark_binds_admission_and_resume_not_growth, tp.test_incremental_fork_copies_on_demand,
            tp.test_preempted_prefix_blocks_stay_cached]
    pins += [lambda s=s: tp.test_hits_match_brute_force(s) for s in range(3)]
    return pins


def test_block_local_cache_key_is_caught(monkeypatch):
    # planted: a block keyed by its own tokens only, not by the prefix it ends
    monkeypatch.setattr(bmod.BlockManager, "_block_key", lambda self, t, i: tuple(t[self.b * i: self.b * (i + 1)]))
    assert _fails(_policy_pins()) >= 1


def test_plain_lru_eviction_is_caught(monkeypatch):
    def victim(self):  # planted: evicts an idle block that cached blocks still extend
        idle = [blk for blk in self.key if self.ref[blk] == 0]
        return min(idle, key=lambda blk: (self.last_use[blk], blk))

    monkeypatch.setattr(bmod.BlockManager, "_victim", victim)
    assert _fails(_policy_pins()) >= 1


def test_most_recent_eviction_is_caught(monkeypatch):
    def victim(self):  # planted: most recently released leaf
        leaves = [blk for blk in self.key if self.ref[blk] == 0 and self.children.get(blk, 0) == 0]
        return max(leaves, key=lambda blk: (self.last_use[blk], blk))

    monkeypatch.setattr(bmod.BlockManager, "_victim", victim)
    assert _fails(_policy_pins()) >= 1


def test_counting_reused_idle_blocks_as_room_is_caught(monkeypatch):
    monkeypatch.setattr(bmod.BlockManager, "_room", lambda self, hits: self.available())
    assert _fails(_policy_pins()) >= 1


def test_ignored_watermark_is_caught(monkeypatch):
    real = bmod.BlockManager.__init__

    def init(self, *a, **kw):
        real(self, *a, **kw)
        self.watermark = 0  # planted

    monkeypatch.setattr(bmod.BlockManager, "__init__", init)
    assert _fails(_policy_pins()) >= 1


def test_incremental_reserving_the_output_is_caught(monkeypatch):
    real = bmod.BlockManager.admit

    def admit(self, prompt_len, max_new, group=-1, prefix_len=0, tokens=None):
        inc = self.incremental
        self.incremental = False  # planted: admission charges the output too
        try:
            return real(self, prompt_len, max_new, group, prefix_len, tokens)
        finally:
            self.incremental = inc

    monkeypatch.setattr(bmod.BlockManager, "admit", admit)
    assert _fails(_policy_pins()) >= 1


def test_preemption_that_drops_tokens_is_caught(monkeypatch):
    real = bmod.BlockManager.preempt

    def preempt(self, sid):
        n = real(self, sid)
        self.seqs[sid].ctx = 0  # planted: the sequence restarts from nothing
        return n

    monkeypatch.setattr(bmod.BlockManager, "preempt", preempt)
    assert _fails(_policy_pins()) >= 1
