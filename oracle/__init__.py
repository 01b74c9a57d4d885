"""Oracle for paged decode attention, KV append, block copy and block accounting.

TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline leg may import this package. The product path never calls it and
shares no code with it.

Plain, slow CPU code that restates what the pages define:
  - paged_attention: softmax(scale * q K^T) V over a context gathered through a
    block table, in float64 from exactly widened bf16 inputs;
  - cache_ops: the slot arithmetic of the block table, append and block copy;
  - block_manager: free list, refcounts, copy-on-write and page-rounded
    admission with full output reservation;
  - accounting: the pages' closed-form memory arithmetic;
  - scenario: replays a workload's events with the pieces above.

Parity pins: every function here is pinned by tests/test_oracle_*.py against
the pages' worked numbers, closed forms, invariants or an independent library
routine (torch's scaled_dot_product_attention in float64).
"""
from . import accounting, block_manager, cache_ops, paged_attention, scenario  # noqa: F401
