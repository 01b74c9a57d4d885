"""ctypes binding of libpkv (include/pkv.h): argument marshalling only.

Every operation runs in the library's CUDA kernels or its C++ block manager;
torch is used for device memory, streams and dtype views. Importing this
module fails loudly if libpkv.so has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpkv.so")

PKV_OK = 0
PKV_EINVAL = -1
PKV_ENOMEM = -2
PKV_ERANGE = -3
PKV_ECUDA = -4
PKV_ENOSPC = -5
PKV_EUNSUPPORTED = -6
PKV_ESTATE = -7

DEVERR_BLOCK_ID = 0x1
DEVERR_SLOT = 0x2
DEVERR_CONTEXT = 0x4
DEVERR_TIMEOUT = 0x8

BLOCK_TOKENS = 16
HEAD_DIM = 128
MAX_GROUP = 8
MAX_SEQS = 4096
MAX_CTAS = 2048

EXPORTED = [
    "pkv_version", "pkv_status_string", "pkv_last_cuda_error", "pkv_read_device_error",
    "pkv_append", "pkv_block_copy", "pkv_attn_workspace_size", "pkv_attn_workspace_init",
    "pkv_attn_decode", "pkv_attn_default_ctas", "pkv_bm_create", "pkv_bm_destroy",
    "pkv_bm_admit", "pkv_bm_fork", "pkv_bm_prepare_append", "pkv_bm_free",
    "pkv_bm_block_table", "pkv_bm_context_len", "pkv_bm_batch_tables", "pkv_bm_stats",
    "pkv_bm_refcount", "pkv_attn_decode_static", "pkv_decode_step", "pkv_attn_decode_ex", "pkv_append_ex",
    "pkv_block_copy_ex", "pkv_bm_create_ex", "pkv_bm_admit_tokens", "pkv_bm_preempt", "pkv_bm_resume",
    "pkv_bm_newest_running", "pkv_bm_slots", "pkv_step_layout", "pkv_decode_step_host",
    "pkv_attn_cascade_workspace_size", "pkv_cascade_staging_size", "pkv_cascade_plan", "pkv_attn_decode_cascade",
    "pkv_attn_decode_wait_test", "pkv_attn_decode_cuda_cores", "pkv_attn_workspace_fixed_bytes",
    "pkv_attn_launch_ctas",
]
BLOCK_SIZES = (8, 16, 32, 64)


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = _lib.pkv_status_string(status).decode()
        if status == PKV_ECUDA:
            msg += f" ({_lib.pkv_last_cuda_error().decode()})"
        super().__init__(f"{what}: {msg} [{status}]" if what else f"{msg} [{status}]")


class PoolExhausted(PkvError):
    pass


class ReservationExceeded(PkvError):
    pass


class StatsT(ctypes.Structure):
    _fields_ = [
        ("num_blocks", ctypes.c_int32), ("free_blocks", ctypes.c_int32),
        ("used_blocks", ctypes.c_int32), ("shared_blocks", ctypes.c_int32),
        ("spare_blocks", ctypes.c_int32), ("num_seqs", ctypes.c_int32),
        ("ref_sum", ctypes.c_int64), ("cow_copies", ctypes.c_int64),
        ("cached_blocks", ctypes.c_int32), ("cached_idle_blocks", ctypes.c_int32),
        ("preempted_seqs", ctypes.c_int32), ("available_blocks", ctypes.c_int32),
        ("cache_hits", ctypes.c_int64), ("evictions", ctypes.c_int64),
    ]


class StepLayoutT(ctypes.Structure):
    _fields_ = [(name, ctypes.c_size_t) for name in
                ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens", "src_dst_pairs", "bytes")]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python paged_kv_cache_49_gb300/build.py` "
            "(nvcc for sm_103a); there is no fallback implementation")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    f32 = ctypes.c_float
    sig = {
        "pkv_version": (i32, []),
        "pkv_status_string": (ctypes.c_char_p, [i32]),
        "pkv_last_cuda_error": (ctypes.c_char_p, []),
        "pkv_read_device_error": (i32, [vp, vp, i32, vp]),
        "pkv_append": (i32, [vp, vp, vp, i32, vp, vp, i32, i32, i32, vp, vp]),
        "pkv_block_copy": (i32, [vp, vp, vp, i32, i32, i32, i32, vp, vp]),
        "pkv_append_ex": (i32, [vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, vp, vp]),
        "pkv_block_copy_ex": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp]),
        "pkv_attn_decode_ex": (i32, [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp, vp]),
        "pkv_attn_workspace_size": (sz, [i32, i32]),
        "pkv_attn_workspace_init": (i32, [vp, sz, vp]),
        "pkv_attn_workspace_fixed_bytes": (sz, []),
        "pkv_attn_decode": (i32, [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp, vp]),
        "pkv_attn_default_ctas": (i32, [i32]),
        "pkv_attn_launch_ctas": (i32, [i32, i32, i32, i32]),
        "pkv_attn_decode_cuda_cores": (i32, [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp,
                                             vp]),
        "pkv_attn_decode_wait_test": (i32, [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp,
                                            i32, vp]),
        "pkv_attn_decode_static": (i32, [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, f32, vp, vp, vp]),
        "pkv_decode_step": (i32, [vp, vp, vp, i32, vp, i32, vp, vp, i32, vp, vp, i32, vp, i32, i32, i32, i32,
                                  f32, i32, vp, sz, vp, vp, vp]),
        "pkv_bm_create": (vp, [i32, i32, vp]),
        "pkv_bm_destroy": (None, [vp]),
        "pkv_bm_admit": (i32, [vp, i32, i32, i32, i32, vp]),
        "pkv_bm_fork": (i32, [vp, i32, i32, vp]),
        "pkv_bm_prepare_append": (i32, [vp, vp, i32, vp, vp, vp]),
        "pkv_bm_free": (i32, [vp, i32]),
        "pkv_bm_block_table": (i32, [vp, i32, vp, i32, vp]),
        "pkv_bm_context_len": (i32, [vp, i32, vp]),
        "pkv_bm_batch_tables": (i32, [vp, vp, i32, vp, i32, vp]),
        "pkv_bm_stats": (i32, [vp, vp]),
        "pkv_bm_refcount": (i32, [vp, i32]),
        "pkv_bm_create_ex": (vp, [i32, i32, vp, i32, i32, i32]),
        "pkv_bm_admit_tokens": (i32, [vp, vp, i32, i32, vp, vp]),
        "pkv_bm_preempt": (i32, [vp, i32, vp]),
        "pkv_bm_resume": (i32, [vp, i32]),
        "pkv_bm_newest_running": (i32, [vp]),
        "pkv_bm_slots": (i32, [vp, i32, i32, i32, vp]),
        "pkv_step_layout": (i32, [i32, i32, i32, i32, i32, i32, vp]),
        "pkv_attn_cascade_workspace_size": (sz, [i32, i32, i32, i32, vp, vp]),
        "pkv_cascade_staging_size": (sz, [i32, i32, i32, i32, vp, vp]),
        "pkv_cascade_plan": (i32, [i32, i32, i32, i32, vp, vp, vp, vp, sz, vp, sz, vp]),
        "pkv_attn_decode_cascade": (i32, [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, f32, i32, vp, vp, vp, sz,
                                          vp, vp]),
        "pkv_decode_step_host": (i32, [vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp, vp,
                                       vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    del i64
    return lib


_lib = _load()
lib = _lib


def _check(status: int, what: str) -> None:
    if status == PKV_OK:
        return
    if status == PKV_ENOMEM:
        raise PoolExhausted(status, what)
    if status == PKV_ENOSPC:
        raise ReservationExceeded(status, what)
    raise PkvError(status, what)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, dtype, name: str, cuda: bool = True) -> None:
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ---------------------------------------------------------------------------
# device operations


def new_error_word(device=None) -> torch.Tensor:
    """A zeroed device uint32 error word (held as int32) for append / copy."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def read_device_error(word: torch.Tensor, clear: bool = True, stream=None) -> int:
    host = ctypes.c_uint32(0)
    _check(_lib.pkv_read_device_error(_ptr(word), ctypes.byref(host), int(clear), _stream(stream)),
           "pkv_read_device_error")
    return host.value


def append(k, v, slot_mapping, k_cache, v_cache, device_error=None, stream=None) -> None:
    """Write k[i], v[i] ([T, Hkv, D] bf16) into slot slot_mapping[i] (int64)."""
    _need(k, torch.bfloat16, "k")
    _need(v, torch.bfloat16, "v")
    _need(slot_mapping, torch.int64, "slot_mapping")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    nb, hkv, bt, d = k_cache.shape
    if v_cache.shape != k_cache.shape or bt not in BLOCK_SIZES:
        raise ValueError("caches must be [num_blocks, Hkv, block_tokens in (8, 16, 32, 64), D] and alike")
    T = slot_mapping.numel()
    if k.shape != (T, hkv, d) or v.shape != (T, hkv, d):
        raise ValueError("k, v must be [T, Hkv, D] matching the cache and slot_mapping")
    if bt == BLOCK_TOKENS:
        st = _lib.pkv_append(_ptr(k), _ptr(v), _ptr(slot_mapping), T, _ptr(k_cache), _ptr(v_cache),
                             nb, hkv, d, _ptr(device_error), _stream(stream))
    else:
        st = _lib.pkv_append_ex(_ptr(k), _ptr(v), _ptr(slot_mapping), T, _ptr(k_cache), _ptr(v_cache),
                                nb, hkv, d, bt, _ptr(device_error), _stream(stream))
    _check(st, "pkv_append")


def block_copy(k_cache, v_cache, pairs, device_error=None, stream=None) -> None:
    """Copy physical block pairs[i, 0] onto pairs[i, 1] in both caches."""
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    _need(pairs, torch.int32, "pairs")
    nb, hkv, bt, d = k_cache.shape
    n = pairs.shape[0] if pairs.numel() else 0
    if n and pairs.shape != (n, 2):
        raise ValueError("pairs must be [n, 2]")
    if bt == BLOCK_TOKENS:
        st = _lib.pkv_block_copy(_ptr(k_cache), _ptr(v_cache), _ptr(pairs) if n else None, n, nb, hkv, d,
                                 _ptr(device_error), _stream(stream))
    else:
        st = _lib.pkv_block_copy_ex(_ptr(k_cache), _ptr(v_cache), _ptr(pairs) if n else None, n, nb, hkv, d, bt,
                                    _ptr(device_error), _stream(stream))
    _check(st, "pkv_block_copy")


def default_ctas(num_seqs: int) -> int:
    return int(_lib.pkv_attn_default_ctas(num_seqs))


def launch_ctas(num_seqs: int, num_kv_heads: int, max_blocks_per_seq: int, block_tokens: int = BLOCK_TOKENS) -> int:
    """CTAs attn_decode launches with num_ctas = 0 for this batch shape."""
    return int(_lib.pkv_attn_launch_ctas(num_seqs, num_kv_heads, max_blocks_per_seq, block_tokens))


class AttentionWorkspace:
    """Device scratch for attn_decode: error word, merge counters and per-CTA
    partials, zeroed once at creation. One workspace serves calls of any
    batch and grid whose partial slots fit in it."""

    def __init__(self, num_seqs: int, num_kv_heads: int, device=None, stream=None):
        nbytes = int(_lib.pkv_attn_workspace_size(num_seqs, num_kv_heads))
        if nbytes == 0:
            raise PkvError(PKV_EINVAL, "pkv_attn_workspace_size")
        self.num_seqs, self.num_kv_heads, self.nbytes = num_seqs, num_kv_heads, nbytes
        self.buffer = torch.empty(nbytes + 256, dtype=torch.uint8, device=device or "cuda")
        off = (-self.buffer.data_ptr()) % 256
        self.tensor = self.buffer[off : off + nbytes]
        _check(_lib.pkv_attn_workspace_init(self.tensor.data_ptr(), nbytes, _stream(stream)),
               "pkv_attn_workspace_init")

    @property
    def ptr(self) -> int:
        return self.tensor.data_ptr()

    @staticmethod
    def fixed_bytes() -> int:
        """Leading bytes that must hold zeros between calls (error word,
        merge counters); the rest is scratch."""
        return int(_lib.pkv_attn_workspace_fixed_bytes())

    def error_word(self) -> torch.Tensor:
        return self.tensor[:4].view(torch.int32)

    def read_error(self, clear: bool = True, stream=None) -> int:
        return read_device_error(self.error_word(), clear, stream)


def attn_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out=None, workspace=None,
                num_ctas: int = 0, stream=None):
    """Decode attention through block tables; returns out [B, Hq, 128] bf16."""
    _need(q, torch.bfloat16, "q")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    B, hq, d = q.shape
    nb, hkv, bt, d2 = k_cache.shape
    if d != d2 or v_cache.shape != k_cache.shape or bt not in BLOCK_SIZES:
        raise ValueError("q [B, Hq, D] and caches [NB, Hkv, block_tokens, D] must agree")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables must be [B, W] and context_lens [B]")
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out")
    if workspace is None:
        workspace = AttentionWorkspace(B, hkv, device=q.device, stream=stream)
    if bt == BLOCK_TOKENS:
        st = _lib.pkv_attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                  block_tables.shape[1], _ptr(context_lens), B, hq, hkv, d, nb,
                                  float(scale), int(num_ctas), workspace.ptr, workspace.nbytes,
                                  _ptr(out), _stream(stream))
    else:
        st = _lib.pkv_attn_decode_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                     block_tables.shape[1], _ptr(context_lens), B, hq, hkv, d, nb, bt,
                                     float(scale), int(num_ctas), workspace.ptr, workspace.nbytes,
                                     _ptr(out), _stream(stream))
    _check(st, "pkv_attn_decode")
    return out


def attn_decode_cuda_cores(q, k_cache, v_cache, block_tables, context_lens, scale, out=None, workspace=None,
                           num_ctas: int = 0, stream=None):
    """attn_decode with the per-tile math on the FP32 CUDA cores instead of
    the tensor cores (group sizes 4 and 8, 16-token blocks): the measured
    alternative to the tensor-core kernel."""
    _need(q, torch.bfloat16, "q")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    B, hq, d = q.shape
    nb, hkv, bt, d2 = k_cache.shape
    if d != d2 or v_cache.shape != k_cache.shape or bt != BLOCK_TOKENS:
        raise ValueError("q [B, Hq, D] and caches [NB, Hkv, 16, D] must agree")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables must be [B, W] and context_lens [B]")
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out")
    if workspace is None:
        workspace = AttentionWorkspace(B, hkv, device=q.device, stream=stream)
    _check(_lib.pkv_attn_decode_cuda_cores(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                           block_tables.shape[1], _ptr(context_lens), B, hq, hkv, d, nb,
                                           float(scale), int(num_ctas), workspace.ptr, workspace.nbytes,
                                           _ptr(out), _stream(stream)),
           "pkv_attn_decode_cuda_cores")
    return out


def decode_step(q, k_new, v_new, slot_mapping, pairs, k_cache, v_cache, block_tables, context_lens, scale,
                out, workspace, device_error=None, num_ctas: int = 0, stream=None):
    """One decode step in one library call: block copies (pairs [n, 2]),
    append of k_new / v_new [B, Hkv, D] at slot_mapping, attention -> out."""
    for t, dt, name in ((q, torch.bfloat16, "q"), (k_new, torch.bfloat16, "k_new"),
                        (v_new, torch.bfloat16, "v_new"), (slot_mapping, torch.int64, "slot_mapping"),
                        (pairs, torch.int32, "pairs"), (k_cache, torch.bfloat16, "k_cache"),
                        (v_cache, torch.bfloat16, "v_cache"), (block_tables, torch.int32, "block_tables"),
                        (context_lens, torch.int32, "context_lens"), (out, torch.bfloat16, "out")):
        _need(t, dt, name)
    B, hq, d = q.shape
    nb, hkv, bt, d2 = k_cache.shape
    T = slot_mapping.numel()
    n = pairs.shape[0] if pairs.numel() else 0
    if d != d2 or v_cache.shape != k_cache.shape or bt != BLOCK_TOKENS or out.shape != q.shape:
        raise ValueError("q/out [B, Hq, D] and caches [NB, Hkv, 16, D] must agree")
    if k_new.shape != (T, hkv, d) or v_new.shape != (T, hkv, d) or (n and pairs.shape != (n, 2)):
        raise ValueError("k_new, v_new must be [T, Hkv, D]; pairs [n, 2]")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables must be [B, W] and context_lens [B]")
    _check(_lib.pkv_decode_step(_ptr(k_new), _ptr(v_new), _ptr(slot_mapping), T, _ptr(pairs) if n else None, n,
                                _ptr(k_cache), _ptr(v_cache), nb, _ptr(q), _ptr(block_tables),
                                block_tables.shape[1], _ptr(context_lens), B, hq, hkv, d, float(scale),
                                int(num_ctas), workspace.ptr, workspace.nbytes, _ptr(out), _ptr(device_error),
                                _stream(stream)), "pkv_decode_step")
    return out


def step_layout(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int, max_blocks_per_seq: int,
                num_pairs: int = 0) -> dict:
    """Byte offsets (and total size) of a decode step's inputs in one packed buffer."""
    lay = StepLayoutT()
    _check(_lib.pkv_step_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq, num_pairs,
                                ctypes.byref(lay)), "pkv_step_layout")
    return {name: int(getattr(lay, name)) for name, _ in StepLayoutT._fields_}


def decode_step_host(host_packed, device_staging, num_pairs, k_cache, v_cache, max_blocks_per_seq, num_seqs,
                     num_q_heads, scale, workspace, device_out, host_out, device_error=None, num_ctas: int = 0,
                     stream=None) -> None:
    """pkv_decode_step_host: the packed inputs (uint8 host tensor) staged into
    device memory -- read across the host link by a kernel when pinned, else
    one copy -- then the step, with the output rows written into host_out
    (directly when pinned, else through device_out and one copy)."""
    _need(host_packed, torch.uint8, "host_packed", cuda=False)
    _need(device_staging, torch.uint8, "device_staging")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    _need(device_out, torch.bfloat16, "device_out")
    _need(host_out, torch.bfloat16, "host_out", cuda=False)
    if host_packed.is_cuda or host_out.is_cuda:
        raise ValueError("host_packed and host_out must be host tensors (pinned for asynchronous copies)")
    nb, hkv, bt, d = k_cache.shape
    if bt != BLOCK_TOKENS or v_cache.shape != k_cache.shape:
        raise ValueError("caches must be [NB, Hkv, 16, D] and alike")
    if device_out.shape != (num_seqs, num_q_heads, d) or host_out.shape != device_out.shape:
        raise ValueError("device_out and host_out must be [num_seqs, Hq, D]")
    need = step_layout(num_seqs, num_q_heads, hkv, d, max_blocks_per_seq, num_pairs)["bytes"]
    if host_packed.numel() < need or device_staging.numel() < need:
        raise ValueError(f"packed buffers need {need} bytes")
    _check(_lib.pkv_decode_step_host(_ptr(host_packed), _ptr(device_staging), num_pairs, _ptr(k_cache),
                                     _ptr(v_cache), nb, max_blocks_per_seq, num_seqs, num_q_heads, hkv, d,
                                     float(scale), int(num_ctas), workspace.ptr, workspace.nbytes,
                                     _ptr(device_out), _ptr(host_out), _ptr(device_error), _stream(stream)),
           "pkv_decode_step_host")


class Cascade:
    """Shared-prefix groups of a batch for pkv_attn_decode_cascade: each
    group is (sequence indices of the batch, shared leading blocks). Owns the
    device workspace and the pinned staging of the plan."""

    def __init__(self, num_seqs: int, num_q_heads: int, num_kv_heads: int, groups, device=None, stream=None):
        groups = [(list(map(int, m)), int(sh)) for m, sh in groups]
        self.num_seqs, self.num_q_heads, self.num_kv_heads = num_seqs, num_q_heads, num_kv_heads
        self.groups = groups
        offs = [0]
        for m, _ in groups:
            offs.append(offs[-1] + len(m))
        n = len(groups)
        self._offsets = (ctypes.c_int32 * (n + 1))(*offs)
        self._members = (ctypes.c_int32 * max(1, offs[-1]))(*[x for m, _ in groups for x in m])
        self._shared = (ctypes.c_int32 * max(1, n))(*[sh for _, sh in groups])
        args = (num_seqs, num_q_heads, num_kv_heads, n, self._offsets, self._shared)
        self.nbytes = int(_lib.pkv_attn_cascade_workspace_size(*args))
        staging = int(_lib.pkv_cascade_staging_size(*args))
        if self.nbytes == 0 or staging == 0:
            raise PkvError(PKV_EINVAL, "pkv_attn_cascade_workspace_size")
        self.buffer = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=device or "cuda")
        off = (-self.buffer.data_ptr()) % 256
        self.tensor = self.buffer[off: off + self.nbytes]
        self.staging = torch.empty(staging, dtype=torch.uint8).pin_memory()
        _check(_lib.pkv_attn_workspace_init(self.tensor.data_ptr(), self.nbytes, _stream(stream)),
               "pkv_attn_workspace_init")
        _check(_lib.pkv_cascade_plan(num_seqs, num_q_heads, num_kv_heads, n, self._offsets, self._members, self._shared,
                                     self.tensor.data_ptr(), self.nbytes, self.staging.data_ptr(), staging,
                                     _stream(stream)), "pkv_cascade_plan")

    def decode(self, q, k_cache, v_cache, block_tables, context_lens, scale, out=None, stream=None):
        """Decode attention for the batch the groups describe; returns out."""
        _need(q, torch.bfloat16, "q")
        _need(k_cache, torch.bfloat16, "k_cache")
        _need(v_cache, torch.bfloat16, "v_cache")
        _need(block_tables, torch.int32, "block_tables")
        _need(context_lens, torch.int32, "context_lens")
        B, hq, d = q.shape
        nb, hkv, bt, _ = k_cache.shape
        if (B, hq, hkv) != (self.num_seqs, self.num_q_heads, self.num_kv_heads) or bt != BLOCK_TOKENS:
            raise ValueError("batch shape differs from the plan's, or blocks are not 16 tokens")
        if out is None:
            out = torch.empty_like(q)
        _need(out, torch.bfloat16, "out")
        _check(_lib.pkv_attn_decode_cascade(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                            block_tables.shape[1], _ptr(context_lens), B, hq, hkv, d, nb,
                                            float(scale), len(self.groups), self._offsets, self._shared,
                                            self.tensor.data_ptr(), self.nbytes, _ptr(out), _stream(stream)),
               "pkv_attn_decode_cascade")
        return out

    def read_error(self, clear: bool = True, stream=None) -> int:
        """The device error word the three kernels share (then cleared)."""
        return read_device_error(self.tensor[:4].view(torch.int32), clear, stream)


def attn_decode_static(q, k_cache, v_cache, block_tables, context_lens, scale, out, device_error=None,
                       stream=None):
    """attn_decode without a workspace, for callers that cannot allocate:
    the library's own static device scratch is used and nothing is allocated
    (out must be given). Calls on one device must not overlap on the GPU."""
    _need(q, torch.bfloat16, "q")
    _need(k_cache, torch.bfloat16, "k_cache")
    _need(v_cache, torch.bfloat16, "v_cache")
    _need(block_tables, torch.int32, "block_tables")
    _need(context_lens, torch.int32, "context_lens")
    _need(out, torch.bfloat16, "out")
    B, hq, d = q.shape
    nb, hkv, bt, d2 = k_cache.shape
    if d != d2 or v_cache.shape != k_cache.shape or bt != BLOCK_TOKENS or out.shape != q.shape:
        raise ValueError("q/out [B, Hq, D] and caches [NB, Hkv, 16, D] must agree")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables must be [B, W] and context_lens [B]")
    _check(_lib.pkv_attn_decode_static(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                       block_tables.shape[1], _ptr(context_lens), B, hq, hkv, d, nb,
                                       float(scale), _ptr(device_error), _ptr(out), _stream(stream)),
           "pkv_attn_decode_static")
    return out


# ---------------------------------------------------------------------------
# host block manager


class BlockManager:
    """Free list, refcounts, copy-on-write, page-rounded admission, incremental
    allocation with preemption, and the prefix-cache index (C++)."""

    def __init__(self, num_blocks: int, block_tokens: int = BLOCK_TOKENS, free_order=None,
                 incremental: bool = False, watermark: int = 0, prefix_cache: bool = False):
        order = None
        self._order_buf = None
        if free_order is not None:
            arr = (ctypes.c_int32 * num_blocks)(*[int(x) for x in free_order])
            self._order_buf = arr
            order = ctypes.cast(arr, ctypes.c_void_p)
        self._h = _lib.pkv_bm_create_ex(num_blocks, block_tokens, order, int(incremental), watermark,
                                        int(prefix_cache))
        if not self._h:
            raise PkvError(PKV_EINVAL, "pkv_bm_create_ex")
        self.num_blocks = num_blocks
        self.reused: dict[int, int] = {}

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            _lib.pkv_bm_destroy(h)
            self._h = None

    def admit(self, prompt_len: int, max_new: int, group: int = -1, prefix_len: int = 0, tokens=None) -> int:
        """tokens (the prompt's ids) selects pkv_bm_admit_tokens; the number of
        reused cached blocks is then kept in self.reused[seq_id]."""
        sid = ctypes.c_int(0)
        if tokens is None:
            _check(_lib.pkv_bm_admit(self._h, prompt_len, max_new, group, prefix_len, ctypes.byref(sid)),
                   "pkv_bm_admit")
            self.reused[sid.value] = 0
            return sid.value
        if group >= 0 or len(tokens) != prompt_len:
            raise PkvError(PKV_EINVAL, "pkv_bm_admit_tokens: no group, one token per prompt position")
        buf = (ctypes.c_int32 * max(prompt_len, 1))(*[int(t) for t in tokens])
        reused = ctypes.c_int(0)
        _check(_lib.pkv_bm_admit_tokens(self._h, buf, prompt_len, max_new, ctypes.byref(sid),
                                        ctypes.byref(reused)), "pkv_bm_admit_tokens")
        self.reused[sid.value] = reused.value
        return sid.value

    def fork(self, parent: int, n: int) -> list[int]:
        ids = (ctypes.c_int32 * max(n, 1))()
        _check(_lib.pkv_bm_fork(self._h, parent, n, ids), "pkv_bm_fork")
        return list(ids[:n])

    def prepare_append(self, seq_ids):
        """Returns (slots list[int], pairs list[(src, dst)])."""
        n = len(seq_ids)
        ids = (ctypes.c_int32 * max(n, 1))(*seq_ids)
        slots = (ctypes.c_int64 * max(n, 1))()
        pairs = (ctypes.c_int32 * max(2 * n, 2))()
        npairs = ctypes.c_int(0)
        _check(_lib.pkv_bm_prepare_append(self._h, ids, n, slots, pairs, ctypes.byref(npairs)),
               "pkv_bm_prepare_append")
        return list(slots[:n]), [(pairs[2 * i], pairs[2 * i + 1]) for i in range(npairs.value)]

    def free(self, seq_id: int) -> None:
        _check(_lib.pkv_bm_free(self._h, seq_id), "pkv_bm_free")
        self.reused.pop(seq_id, None)

    def preempt(self, seq_id: int) -> int:
        n = ctypes.c_int(0)
        _check(_lib.pkv_bm_preempt(self._h, seq_id, ctypes.byref(n)), "pkv_bm_preempt")
        return n.value

    def resume(self, seq_id: int) -> None:
        _check(_lib.pkv_bm_resume(self._h, seq_id), "pkv_bm_resume")

    def newest_running(self) -> int:
        return int(_lib.pkv_bm_newest_running(self._h))

    def slots(self, seq_id: int, first: int, n: int) -> list[int]:
        buf = (ctypes.c_int64 * max(n, 1))()
        _check(_lib.pkv_bm_slots(self._h, seq_id, first, n, buf), "pkv_bm_slots")
        return list(buf[:n])

    def table(self, seq_id: int) -> list[int]:
        length = ctypes.c_int(0)
        st = _lib.pkv_bm_block_table(self._h, seq_id, None, 0, ctypes.byref(length))
        if st not in (PKV_OK, PKV_ERANGE):
            _check(st, "pkv_bm_block_table")
        buf = (ctypes.c_int32 * max(length.value, 1))()
        _check(_lib.pkv_bm_block_table(self._h, seq_id, buf, length.value, ctypes.byref(length)),
               "pkv_bm_block_table")
        return list(buf[: length.value])

    def context_len(self, seq_id: int) -> int:
        c = ctypes.c_int(0)
        _check(_lib.pkv_bm_context_len(self._h, seq_id, ctypes.byref(c)), "pkv_bm_context_len")
        return c.value

    def batch_tables(self, seq_ids, width: int):
        """(tables int32 [n, width] with -1 padding, context_lens int32 [n]) as CPU tensors."""
        n = len(seq_ids)
        ids = (ctypes.c_int32 * max(n, 1))(*seq_ids)
        tables = torch.empty((n, width), dtype=torch.int32)
        ctx = torch.empty((n,), dtype=torch.int32)
        _check(_lib.pkv_bm_batch_tables(self._h, ids, n, tables.data_ptr(), width, ctx.data_ptr()),
               "pkv_bm_batch_tables")
        return tables, ctx

    def stats(self) -> dict:
        s = StatsT()
        _check(_lib.pkv_bm_stats(self._h, ctypes.byref(s)), "pkv_bm_stats")
        return {"free": s.free_blocks, "used": s.used_blocks, "shared": s.shared_blocks,
                "ref_sum": s.ref_sum, "spares": s.spare_blocks, "cow_copies": s.cow_copies,
                "seqs": s.num_seqs, "cached": s.cached_blocks, "cached_idle": s.cached_idle_blocks,
                "available": s.available_blocks, "cache_hits": s.cache_hits, "evictions": s.evictions,
                "preempted": s.preempted_seqs}

    def refcount(self, block: int) -> int:
        return int(_lib.pkv_bm_refcount(self._h, block))
