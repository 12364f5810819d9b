"""The C-ABI library builds, loads without a GPU and exports every entry point the header declares.

No compute call is made here; the only calls are ones that return before touching CUDA
(version, status names, and argument checks that reject a null pool).
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \t\*]*?\b(pkv_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def cdll():
    from paged_kv_attention_10_gb300 import build

    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_hot_path():
    names = declared_functions()
    for n in ("pkv_kv_append", "pkv_paged_gather", "pkv_paged_decode", "pkv_paged_extend",
              "pkv_merge_states", "pkv_decode_workspace_size", "pkv_extend_workspace_size",
              "pkv_status_string", "pkv_version", "pkv_shared_prefix_attention",
              "pkv_shared_prefix_workspace_size", "pkv_merge_states_bf16", "pkv_rope_cos_sin_table",
              "pkv_plan_shared_prefix", "pkv_paged_decode_l2keep"):
        assert n in names


def test_every_declared_symbol_is_exported(cdll):
    missing = [n for n in declared_functions() if not hasattr(cdll, n)]
    assert not missing, f"not exported: {missing}"


def test_host_only_calls(cdll):
    cdll.pkv_version.restype = ctypes.c_int32
    assert cdll.pkv_version() >= 100
    cdll.pkv_status_string.restype = ctypes.c_char_p
    assert cdll.pkv_status_string(0) == b"ok"
    assert cdll.pkv_status_string(3) == b"workspace too small"
    # the bounded-wait check rejects a missing error word before launching anything
    cdll.pkv_selftest_bounded_wait.restype = ctypes.c_int32
    assert cdll.pkv_selftest_bounded_wait(None, None) == 1


def test_null_pool_is_rejected_before_any_cuda_call(cdll):
    INVALID = 1
    f = cdll.pkv_kv_append
    f.restype = ctypes.c_int32
    assert f(None, None, None, None, ctypes.c_int32(1), None, None) == INVALID
    f = cdll.pkv_paged_decode
    f.restype = ctypes.c_int32
    assert f(None, None, ctypes.c_int32(1), ctypes.c_int32(8), None, None, None, ctypes.c_float(1.0),
             None, None, None, ctypes.c_size_t(0), None, None) == INVALID
    f = cdll.pkv_paged_decode_l2keep
    f.restype = ctypes.c_int32
    assert f(None, None, ctypes.c_int32(1), ctypes.c_int32(8), None, None, None, ctypes.c_float(1.0),
             None, None, None, ctypes.c_size_t(0), None, ctypes.c_int32(0), None, None) == INVALID


def test_rope_table_rejects_bad_arguments_before_any_cuda_call(cdll):
    f = cdll.pkv_rope_cos_sin_table
    f.restype = ctypes.c_int32
    f.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_double, ctypes.c_void_p]
    INVALID = 1
    assert f(None, 16, 127, 1e4, None) == INVALID   # odd head_dim
    assert f(None, 16, 128, 0.0, None) == INVALID   # theta must be positive
    assert f(None, -1, 128, 1e4, None) == INVALID   # negative position count
    assert f(None, 16, 128, 1e4, None) == INVALID   # no table
    assert f(None, 0, 128, 1e4, None) == 0          # nothing to build: no launch


class _Sizes(ctypes.Structure):
    _fields_ = [("num_splits", ctypes.c_int32), ("num_parts", ctypes.c_int32),
                ("max_part_rows", ctypes.c_int32), ("num_part_indices", ctypes.c_int32),
                ("num_suffix_indices", ctypes.c_int32)]


def test_plan_shared_prefix_sizes_capacity_and_errors(cdll):
    """The host plan: a size query with no output arrays, PKV_ERR_WORKSPACE (sizes filled) when
    the caller's arrays are too small, and argument errors; counts checked by hand for a batch of
    three requests, the first two sharing two of their pages."""
    import numpy as np

    f = cdll.pkv_plan_shared_prefix
    f.restype = ctypes.c_int32
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p) if a is not None else None
    i32 = lambda v: np.asarray(v, dtype=np.int32)
    indptr, indices, lens = i32([0, 3, 6, 8]), i32([7, 8, 1, 7, 8, 2, 5, 6]), i32([40, 37, 20])
    gf, gc = i32([0]), i32([2])
    sz = _Sizes()

    def call(*outs, parts_cap=0, idx_cap=0, groups=(gf, gc, 1), ps=16):
        return f(p(indptr), p(indices), p(lens), 3, p(groups[0]), p(groups[1]), groups[2], ps, 2, 4, 152,
                 2, 16, ctypes.byref(sz), *[p(o) for o in outs], parts_cap, idx_cap)

    assert call(*([None] * 10)) == 0
    # two shared pages (32 positions, each member keeps one own position), chunks of >= 16
    # positions: S = 2; parts: the group's 2 chunks and 2 empty parts for the third request
    assert (sz.num_splits, sz.num_parts, sz.max_part_rows) == (2, 4, 2)
    assert (sz.num_part_indices, sz.num_suffix_indices) == (2, 4)
    shared = np.zeros(1, np.int32)
    arrs = [np.zeros(n, np.int32) for n in (4, 4, 4, 5, 8, 4, 4, 8, 3)]
    assert call(shared, *[a[:1] for a in arrs], parts_cap=1, idx_cap=8) == 3  # too small a capacity
    assert sz.num_parts == 4
    assert call(shared, *arrs, parts_cap=4, idx_cap=8) == 0
    q_start, q_len, o_start, p_indptr, p_indices, p_lens, s_indptr, s_indices, s_lens = arrs
    assert shared[0] == 32
    assert q_start.tolist() == [0, 0, 2, 2] and q_len.tolist() == [2, 2, 1, 1]
    assert o_start.tolist() == [0, 3, 2, 5]
    assert p_indptr.tolist() == [0, 1, 2, 2, 2] and p_indices[:2].tolist() == [7, 8]
    assert p_lens.tolist() == [16, 16, 0, 0]
    assert s_indptr.tolist() == [0, 1, 2, 4] and s_indices[:4].tolist() == [1, 2, 5, 6]
    assert s_lens.tolist() == [8, 5, 20]
    # a group past the batch, overlapping groups, a bad page size
    assert call(*([None] * 10), groups=(i32([2]), i32([2]), 1)) == 1
    assert call(*([None] * 10), groups=(i32([0, 1]), i32([2, 2]), 2)) == 1
    assert call(*([None] * 10), ps=0) == 1
