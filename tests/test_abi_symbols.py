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
              "pkv_plan_shared_prefix"):
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
