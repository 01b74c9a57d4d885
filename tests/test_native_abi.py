"""The C-ABI library loads and exports every function include/pkv.h declares
(no compute calls: these run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib_path():
    from tests.conftest import build_native
    return build_native()


def _declared():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("pkv_append", "pkv_attn_decode", "pkv_block_copy", "pkv_bm_admit",
                     "pkv_bm_prepare_append", "pkv_bm_free"):
        assert required in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_the_header(lib_path):
    import paged_kv_cache_49_gb300 as pkv
    assert sorted(pkv.EXPORTED) == _declared()


def test_version_and_status_strings(lib_path):
    import paged_kv_cache_49_gb300._native as nat
    assert nat.lib.pkv_version() == 100
    assert nat.lib.pkv_status_string(nat.PKV_ENOMEM) == b"too few free pages"
    assert nat.lib.pkv_status_string(12345) == b"unknown status"


def test_host_argument_checks_need_no_gpu(lib_path):
    import paged_kv_cache_49_gb300._native as nat
    L = nat.lib
    # null pointers and bad shapes are rejected before any CUDA call
    assert L.pkv_attn_decode(None, None, None, None, 1, None, 1, 32, 8, 128, 1, 1.0, 0, None, 0, None, None) == nat.PKV_EINVAL
    assert L.pkv_append(None, None, None, -1, None, None, 1, 8, 128, None, None) == nat.PKV_EINVAL
    assert L.pkv_append(None, None, None, 0, None, None, 1, 8, 128, None, None) == nat.PKV_OK
    assert L.pkv_block_copy(None, None, None, 0, 1, 8, 128, None, None) == nat.PKV_OK
    assert L.pkv_block_copy(None, None, None, 3, 1, 8, 127, None, None) == nat.PKV_EINVAL
    assert L.pkv_attn_workspace_size(0, 8) == 0
    assert L.pkv_bm_create(0, 16, None) is None
    assert L.pkv_bm_create(4, 12, None) is None  # block sizes are 8, 16, 32 or 64
    h = L.pkv_bm_create(4, 8, None)
    assert h is not None
    L.pkv_bm_destroy(h)
    assert L.pkv_attn_decode_ex(None, None, None, None, 1, None, 1, 32, 8, 128, 1, 16, 1.0, 0, None, 0, None, None) == nat.PKV_EINVAL


def test_step_layout_is_packed_and_aligned(lib_path):
    import paged_kv_cache_49_gb300._native as nat
    B, hq, hkv, d, w = 5, 32, 8, 128, 37
    order = ["q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens", "src_dst_pairs"]
    sizes = {"q": B * hq * d * 2, "k_new": B * hkv * d * 2, "v_new": B * hkv * d * 2, "slot_mapping": B * 8,
             "block_tables": B * w * 4, "context_lens": B * 4}
    for pairs in (0, 3):
        lay = nat.step_layout(B, hq, hkv, d, w, pairs)
        sizes["src_dst_pairs"] = pairs * 8
        end = 0
        for name in order:
            assert lay[name] % 256 == 0 and lay[name] >= end
            end = lay[name] + sizes[name]
        assert lay["bytes"] >= end and lay["bytes"] - end < 256
    assert nat.step_layout(B, hq, hkv, d, w, 0)["context_lens"] == nat.step_layout(B, hq, hkv, d, w, 9)["context_lens"]
    lay = nat.StepLayoutT()
    assert nat.lib.pkv_step_layout(0, 32, 8, 128, 1, 0, ctypes.byref(lay)) == nat.PKV_EINVAL
    assert nat.lib.pkv_decode_step_host(None, None, 0, None, None, 1, 1, 1, 32, 8, 128, 1.0, 0, None, 0, None,
                                        None, None, None) == nat.PKV_EINVAL
