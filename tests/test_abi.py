"""The C-ABI library builds for sm_103a, loads, exports every symbol that
include/csa2.h declares, and rejects bad arguments on the host before any GPU
work (these calls return before touching a device, so they run without one)."""
import ctypes
import os
import re

import pytest

import sparse_attention_decode_step_gb300 as csa
from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "csa2.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    L = csa.lib()
    names = _declared()
    assert "csa2_sparse_attn" in names and len(names) >= 13
    for n in names:
        assert hasattr(L, n), n
    assert set(csa.EXPORTS) == set(names)


def test_built_for_sm103a_only():
    from sparse_attention_decode_step_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert os.path.exists(csa.library_path())


def test_status_strings():
    L = csa.lib()
    for code in (0, -1, -2, -3, -4, -5):
        assert L.csa2_status_string(code)


def test_workspace_sizes_are_host_only_and_monotone():
    a = csa.index_workspace_size(32, 1, 8, 128)
    b = csa.index_workspace_size(64, 1, 8, 128)
    assert 0 < a < b
    assert csa.index_workspace_size(33, 2, 8, 128) == 0          # nq not a multiple of group
    t1 = csa.topk_workspace_size(8, 16384)
    t2 = csa.topk_workspace_size(8, 1 << 20)
    assert 0 < t1 < t2
    # the attention's splits merge inside a thread-block cluster: no workspace
    assert csa.attn_workspace_size(32, 64, 2048, 128) == 0
    assert csa.attn_workspace_size(1, 64, 16384, 128) == 0


def _cache(**over):
    c = csa._Cache(16, 16, 16, 16, 16, 16, 64, 1, 128, 1)
    for k, v in over.items():
        setattr(c, k, v)
    return c


def test_append_rejects_bad_arguments_on_host():
    L = csa.lib()
    ok_ptr = ctypes.c_void_p(4096)
    c = _cache()
    # n_tok not a multiple of m
    c2 = _cache(m=2)
    assert L.csa2_quantize_append(ctypes.byref(c2), ok_ptr, ok_ptr, ok_ptr, 3, None, None) == -1
    # unsupported d_idx
    c3 = _cache(d_idx=96)
    assert L.csa2_quantize_append(ctypes.byref(c3), ok_ptr, None, ok_ptr, 1, None, None) == -4
    # misaligned latent pointer
    assert L.csa2_quantize_append(ctypes.byref(c), ctypes.c_void_p(4100), None, ok_ptr, 1, None,
                                  None) == -2
    # NULL cache
    assert L.csa2_quantize_append(None, ok_ptr, None, ok_ptr, 1, None, None) == -1
    # the projecting append: w_ik required and 16-byte aligned, same cache checks
    assert L.csa2_quantize_append_project(ctypes.byref(c), ok_ptr, None, None, 1, None, None) == -1
    assert L.csa2_quantize_append_project(ctypes.byref(c), ok_ptr, None, ctypes.c_void_p(4100), 1,
                                          None, None) == -2
    assert L.csa2_quantize_append_project(ctypes.byref(c3), ok_ptr, None, ok_ptr, 1, None,
                                          None) == -4
    # capacity must be a multiple of 8
    c4 = _cache(cap=60)
    assert L.csa2_quantize_append(ctypes.byref(c4), ok_ptr, None, ok_ptr, 1, None, None) == -1


def test_index_rejects_bad_arguments_on_host():
    L = csa.lib()
    p = ctypes.c_void_p(4096)
    c = _cache()
    q = csa._Queries(4096, 4096, 4, 1)
    # h_idx too large
    assert L.csa2_index_full(ctypes.byref(c), ctypes.byref(q), p, p, 17, 64, p, 64, None, 0, None,
                             p, 1 << 20, None, None) == -4
    # ld_scores < max_n
    assert L.csa2_index_full(ctypes.byref(c), ctypes.byref(q), p, p, 8, 128, p, 64, None, 0, None,
                             p, 1 << 20, None, None) == -1
    # workspace too small
    assert L.csa2_index_full(ctypes.byref(c), ctypes.byref(q), p, p, 8, 64, p, 64, None, 0, None,
                             p, 16, None, None) == -3
    # group must divide nq
    q2 = csa._Queries(4096, 4096, 4, 3)
    assert L.csa2_index_full(ctypes.byref(c), ctypes.byref(q2), p, p, 8, 64, p, 64, None, 0, None,
                             p, 1 << 20, None, None) == -1
    # Reindex needs group 1 and a pool
    assert L.csa2_index_reindex(ctypes.byref(c), ctypes.byref(q), p, p, 8, None, None, 2048, p,
                                16384, None, p, 1 << 20, None, None) == -1
    # zero queries is a no-op
    q0 = csa._Queries(None, None, 0, 1)
    assert L.csa2_index_full(ctypes.byref(c), ctypes.byref(q0), p, p, 8, 64, p, 64, None, 0, None,
                             p, 1 << 20, None, None) == 0


def test_topk_attn_layer_reject_bad_arguments_on_host():
    L = csa.lib()
    p = ctypes.c_void_p(4096)
    assert L.csa2_topk(p, 64, p, None, 0, 2, 128, 8, p, 8, p, p, 1 << 20, None) == -1   # ld < max_n
    assert L.csa2_topk(p, 66, p, None, 0, 2, 64, 8, p, 8, p, p, 1 << 20, None) == -1    # ld % 4
    assert L.csa2_topk(p, 64, p, None, 0, 2, 64, 0, p, 8, p, p, 1 << 20, None) == -1    # k = 0
    assert L.csa2_topk(p, 64, p, None, 0, 2, 64, 8, p, 8, p, p, 8, None) == -3          # workspace
    assert L.csa2_topk(p, 64, p, None, 0, 0, 64, 8, p, 8, p, p, 8, None) == 0           # nq = 0
    c = _cache()
    q = csa._Queries(4096, 4096, 4, 1)
    # H out of range
    assert L.csa2_sparse_attn(ctypes.byref(c), ctypes.byref(q), p, 8, p, 8, p, 65, p, 128, None,
                              128, 1.0, p, None, p, 1 << 30, None, None) == -4
    # window ring smaller than the window
    assert L.csa2_sparse_attn(ctypes.byref(c), ctypes.byref(q), p, 8, p, 8, p, 16, p, 64, None,
                              128, 1.0, p, None, p, 1 << 30, None, None) == -1
    a = csa._LayerArgs()
    a.mode = 7
    assert L.csa2_layer_step(ctypes.byref(a), None) == -1
    assert L.csa2_layer_step(None, None) == -1


def test_launch_counter_starts_readable():
    assert csa.launch_count() >= 0
