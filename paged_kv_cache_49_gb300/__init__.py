"""GB300-native paged KV cache decode.

libpkv (C ABI, include/pkv.h) holds the CUDA kernels for sm_103a -- paged
decode attention, KV append, copy-on-write block copy -- and the C++ host
block manager. This package is the thin Python binding over it plus a small
engine that drives one attention layer's pool.
"""
from ._native import (  # noqa: F401
    BLOCK_TOKENS, DEVERR_BLOCK_ID, DEVERR_CONTEXT, DEVERR_SLOT, DEVERR_TIMEOUT, EXPORTED,
    HEAD_DIM, LIB_PATH, MAX_CTAS, MAX_GROUP, AttentionWorkspace, BlockManager, Cascade, PkvError, PoolExhausted,
    ReservationExceeded, append, attn_decode, attn_decode_cuda_cores, attn_decode_static, block_copy, decode_step, decode_step_host,
    default_ctas, launch_ctas, new_error_word, step_layout,
    read_device_error,
)
from .engine import (  # noqa: F401
    CASCADE_MIN_SAVED_BYTES, HostStep, PagedKVEngine, StepBuffers, bf16_from_bits, bits_from_bf16, cascade_saved_bytes,
    shared_prefix_groups,
)
from .graphs import GraphedDecoder, default_buckets  # noqa: F401
