"""The pages' closed-form KV memory arithmetic.

  - "KV cache systems", kv bytes/token equation:
        kv = 2 * n_layers * n_kv * d_h * bytes_per_element
  - "Reserve the page a request has not written yet", "Separate the pool from
    its owners": page bytes = tokens per page * kv; pool pages = pool bytes /
    page bytes; request pages = ceil((prompt + output) / 16).
  - "Charge shared pages once": a group of requests sharing complete prefix
    pages needs shared + sum of private pages.
  - "KV cache systems", last-block paragraph: a request of D tokens holds
    ceil(D / b) blocks and wastes b * ceil(D / b) - D tokens.
"""
from __future__ import annotations


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, bytes_per_elem: int = 2) -> int:
    return 2 * n_layers * n_kv_heads * head_dim * bytes_per_elem


def page_bytes(tokens_per_page: int, kv_per_token: int) -> int:
    return tokens_per_page * kv_per_token


def pool_pages(pool_bytes: int, page: int) -> int:
    return pool_bytes // page


def request_pages(prompt_len: int, max_output: int, tokens_per_page: int = 16) -> int:
    return ceil_div(prompt_len + max_output, tokens_per_page)


def group_pages(n_requests: int, prefix_len: int, suffix_len: int, tokens_per_page: int = 16) -> int:
    """Pages for n requests that share the complete pages of one prefix."""
    shared = prefix_len // tokens_per_page
    private = request_pages(prefix_len, suffix_len, tokens_per_page) - shared
    return shared + n_requests * private


def max_admitted(pool: int, first_cost: int, next_cost: int) -> int:
    """How many requests fit when the first costs first_cost pages and each
    further one next_cost (next_cost == first_cost when nothing is shared)."""
    if first_cost > pool:
        return 0
    return 1 + (pool - first_cost) // next_cost


def tail_waste(tokens: int, tokens_per_page: int = 16) -> int:
    return tokens_per_page * ceil_div(tokens, tokens_per_page) - tokens


def table_entries(tokens: int, tokens_per_page: int = 16) -> int:
    return ceil_div(tokens, tokens_per_page)
