"""The C ABI: libpkv.so builds for sm_103a, loads without a GPU, exports every
symbol include/pkv.h declares, and rejects bad host arguments before any
CUDA call (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import paged_kv_decode_pages_gb300 as pkv
from paged_kv_decode_pages_gb300 import _binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _binding.load()


def test_header_declares_the_four_entry_points():
    names = _declared()
    for fn in ("pkv_kv_append", "pkv_paged_decode_attn", "pkv_seeded_sample",
               "pkv_codebook_frame_sample"):
        assert fn in names


def test_every_declared_symbol_is_exported_and_bound(lib):
    names = _declared()
    assert set(names) == set(_binding.SIGNATURES)
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_error_strings(lib):
    assert "sm_103a" in pkv.version()
    assert pkv.error_string(0) == "ok"
    assert "workspace" in pkv.error_string(4)
    assert lib.pkv_num_dev_error_bits() == 7
    # a CUDA failure is named by the runtime's own error names (host only)
    assert lib.pkv_cuda_error_name(700) == b"cudaErrorIllegalAddress"
    assert lib.pkv_cuda_error_name(716) == b"cudaErrorMisalignedAddress"


def test_workspace_sizes_are_host_only(lib):
    # long-context shape: 16 rows, 32 q heads, head_dim 128, 2048 pages
    ws = pkv.decode_workspace_bytes(16, 32, 128, 2048)
    assert ws >= 16 * 32 * 64 * (128 + 2) * 4
    assert pkv.decode_workspace_bytes(0, 32, 128, 2048) == 0
    assert pkv.sample_workspace_bytes(16, 151936) > 0
    assert pkv.frame_workspace_bytes(12, 32, 1024) >= 32 * 1024 * 4


def test_host_validation_rejects_before_launch(lib):
    g = _binding.pkv_cache_t(1, 4, 16, 2, 64)
    P = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    st = lib.pkv_kv_append(None, P, 0, P, P, P, 1, P, P, 1, None, None)
    assert st == 1
    st = lib.pkv_kv_append(ctypes.byref(g), P, 5, P, P, P, 1, P, P, 1, None, None)  # bad layer
    assert st == 1
    st = lib.pkv_paged_decode_attn(ctypes.byref(g), P, 0, P, 3, 1.0, P, 1, P, P, 1, P, 0, None,
                                   None, 0, None, None)  # 3 q heads over 2 kv heads
    assert st == 1
    g2 = _binding.pkv_cache_t(1, 4, 16, 2, 96)  # head_dim 96
    st = lib.pkv_paged_decode_attn(ctypes.byref(g2), P, 0, P, 4, 1.0, P, 1, P, P, 1, P, 0, None,
                                   None, 0, None, None)
    assert st == 2
    g3 = _binding.pkv_cache_t(1, 4, 16, 2, 64)
    st = lib.pkv_paged_decode_attn(ctypes.byref(g3), P, 0, P, 4, 1.0, P, 100, P, P, 1, P, 0, None,
                                   None, 0, None, None)  # 4 splits, no workspace
    assert st == 4
    # the plan / planned pair: the same checks as the per-call entry point
    st = lib.pkv_decode_plan(ctypes.byref(g3), 4, 100, P, P, 1, None, 0, None, None)
    assert st == 4  # no workspace
    st = lib.pkv_decode_plan(ctypes.byref(g3), 4, 100, None, P, 1, P, 1 << 20, None, None)
    assert st == 1  # no seq_lens
    st = lib.pkv_decode_plan(ctypes.byref(g3), 3, 100, P, P, 1, P, 1 << 20, None, None)
    assert st == 1  # 3 q heads over 2 kv heads
    st = lib.pkv_paged_decode_attn_planned(ctypes.byref(g2), P, 0, P, 4, 1.0, P, 1, P, P, 1, P,
                                           0, None, None, 0, None, None)
    assert st == 2  # head_dim 96
    st = lib.pkv_paged_decode_attn_planned(ctypes.byref(g3), P, 0, P, 4, 1.0, P, 100, P, P, 1,
                                           P, 0, None, None, 0, None, None)
    assert st == 4  # no workspace
    # the static-scratch form: argument errors are named whatever the size,
    # and an oversized problem is refused before any CUDA call
    big = 1 << 20  # max_pages: far more scratch than the library's array
    st = lib.pkv_paged_decode_attn_static(ctypes.byref(g2), P, 0, P, 4, 1.0, P, big, P, P, 64, P,
                                          0, None, None, None)
    assert st == 2  # head_dim 96, not "workspace too small"
    st = lib.pkv_paged_decode_attn_static(ctypes.byref(g3), P, 0, P, 3, 1.0, P, big, P, P, 64, P,
                                          0, None, None, None)
    assert st == 1  # 3 q heads over 2 kv heads
    st = lib.pkv_paged_decode_attn_static(ctypes.byref(g3), P, 0, None, 4, 1.0, P, big, P, P, 64,
                                          P, 0, None, None, None)
    assert st == 1  # no q
    st = lib.pkv_paged_decode_attn_static(ctypes.byref(g3), P, 0, P, 4, 1.0, P, big, P, P, 64, P,
                                          0, None, None, None)
    assert st == 4  # well-formed, larger than the array
    assert lib.pkv_selftest_wait_timeout(0, P, None) == 1  # no limit
    assert lib.pkv_selftest_wait_timeout(2 * 10**9, P, None) == 1  # over a second
    assert lib.pkv_selftest_wait_timeout(1000, None, None) == 1  # no error word
    st = lib.pkv_seeded_sample(P, 16, 1, 16, P, P, 1, P, P, P, P, P, 0, 1, None, 0, 0, 0, P, P,
                               None, 0, None, None)  # no workspace
    assert st == 4
    st = lib.pkv_seeded_sample(P, 8, 1, 16, P, P, 1, P, P, P, P, P, 0, 1, None, 0, 0, 0, P, P,
                               None, 0, None, None)  # row_stride < vocab
    assert st == 1
    st = lib.pkv_codebook_frame_sample(P, None, 0, 1, 16, P, P, 1, P, P, P, P, P, P, P, P, 1 << 20,
                                       None, None)  # zero codebooks
    assert st == 1
