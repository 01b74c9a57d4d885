"""Seeded synthetic inputs shared by the tests, the bench and the oracle runs.

This package holds random draws and workload shapes only: no paged-attention,
append, copy or block-accounting arithmetic lives here.
"""
from .gen import (  # noqa: F401
    WORKLOADS,
    Workload,
    bf16_bits,
    make_workload,
    randn_bf16,
)
