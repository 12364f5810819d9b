"""Python binding of libpagedkv (attention over a paged KV pool on GB300).

Argument marshalling only: every function here checks that the tensors it is given have the
dtype, device and contiguity the C ABI expects, passes their device pointers and the current
CUDA stream to the matching ``pkv_*`` entry point, and turns a non-OK status into an exception.
All computation happens in the library's CUDA kernels; there is no CPU or PyTorch fallback, and
a missing library is an error.

Names follow the C ABI in ``include/pagedkv.h`` (``pkv_kv_append`` -> ``kv_append`` ...).
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

__all__ = [
    "load", "library_path", "PagedKVError", "kv_append", "paged_gather", "decode_workspace_size",
    "paged_decode", "paged_decode_noalloc", "extend_workspace_size", "paged_extend",
    "merge_states", "shared_prefix_workspace_size", "shared_prefix_attention", "cascade_decode",
    "status_string", "version", "selftest_bounded_wait", "validate_page_table", "validate_slots",
    "rope_cos_sin_table", "rope_kv_append", "DEVERR_PAGE_OOB", "DEVERR_SLOT_OOB", "DEVERR_LENGTH",
    "DEVERR_TIMEOUT", "DEVERR_INTERNAL", "DEVERR_ROW_OOB",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libpagedkv.so")
_lib = None

DEVERR_PAGE_OOB = 0x1
DEVERR_SLOT_OOB = 0x2
DEVERR_LENGTH = 0x4
DEVERR_TIMEOUT = 0x8
DEVERR_INTERNAL = 0x10
DEVERR_ROW_OOB = 0x20

_c_i32, _c_i64, _c_f32, _c_sz, _vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p


class Pool(ctypes.Structure):
    _fields_ = [("k", _vp), ("v", _vp), ("num_pages", _c_i64), ("page_size", _c_i32),
                ("num_kv_heads", _c_i32), ("head_dim", _c_i32)]


class CascadeSizes(ctypes.Structure):
    _fields_ = [("num_splits", _c_i32), ("num_parts", _c_i32), ("max_part_rows", _c_i32),
                ("num_part_indices", _c_i32), ("num_suffix_indices", _c_i32)]


class PagedKVError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libpagedkv.so (built by ``paged_kv_attention_10_gb300.build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is not built; run paged_kv_attention_10_gb300.build.build()")
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.POINTER(Pool)
    sig = {
        "pkv_status_string": (ctypes.c_char_p, [_c_i32]),
        "pkv_version": (_c_i32, []),
        "pkv_kv_append": (_c_i32, [P, _vp, _vp, _vp, _c_i32, _vp, _vp]),
        "pkv_paged_gather": (_c_i32, [P, _vp, _vp, _vp, _c_i32, _vp, _vp, _vp, _vp]),
        "pkv_decode_workspace_size": (_c_sz, [_c_i32, _c_i32, _c_i32, _c_i32]),
        "pkv_paged_decode": (_c_i32, [P, _vp, _c_i32, _c_i32, _vp, _vp, _vp, _c_f32, _vp, _vp, _vp,
                                      _c_sz, _vp, _vp]),
        "pkv_paged_decode_ctas": (_c_i32, [P, _vp, _c_i32, _c_i32, _vp, _vp, _vp, _c_f32, _vp, _vp,
                                           _vp, _c_sz, _vp, _c_i32, _vp]),
        "pkv_paged_decode_l2keep": (_c_i32, [P, _vp, _c_i32, _c_i32, _vp, _vp, _vp, _c_f32, _vp, _vp,
                                             _vp, _c_sz, _vp, _c_i32, _vp, _vp]),
        "pkv_extend_workspace_size": (_c_sz, [_c_i32, _c_i32, _c_i32, _c_i32, _c_i32]),
        "pkv_paged_extend": (_c_i32, [P, _vp, _c_i32, _vp, _c_i32, _c_i32, _vp, _vp, _vp, _c_i32,
                                      _c_f32, _vp, _vp, _vp, _c_sz, _vp, _vp]),
        "pkv_merge_states": (_c_i32, [_vp, _vp, _c_i32, _c_i32, _c_i32, _c_i32, _vp, _vp, _vp]),
        "pkv_merge_states_bf16": (_c_i32, [_vp, _vp, _c_i32, _c_i32, _c_i32, _c_i32, _vp, _vp, _vp]),
        "pkv_shared_prefix_workspace_size": (_c_sz, [_c_i32, _c_i32, _c_i32, _c_i32, _c_i32]),
        "pkv_shared_prefix_attention": (_c_i32, [P, _vp, _c_i32, _vp, _vp, _vp, _c_i32, _c_i32, _vp, _vp,
                                                 _vp, _c_i32, _c_f32, _vp, _vp, _c_i32, _vp, _c_sz, _vp,
                                                 _vp]),
        "pkv_rope_kv_append": (_c_i32, [P, _vp, _vp, _vp, _vp, _vp, _c_i32, _vp, _c_i32, _c_i32, _vp, _vp]),
        "pkv_paged_decode_noalloc": (_c_i32, [P, _vp, _c_i32, _c_i32, _vp, _vp, _vp, _c_f32, _vp, _vp,
                                              _vp, _vp]),
        "pkv_selftest_bounded_wait": (_c_i32, [_vp, _vp]),
        "pkv_validate_page_table": (_c_i32, [_vp, _vp, _vp, _c_i32, _c_i64, _c_i32, _c_i32, _vp]),
        "pkv_validate_slots": (_c_i32, [_vp, _c_i32, _c_i64, _vp]),
        "pkv_rope_cos_sin_table": (_c_i32, [_vp, _c_i32, _c_i32, ctypes.c_double, _vp]),
        "pkv_plan_shared_prefix": (_c_i32, [_vp, _vp, _vp, _c_i32, _vp, _vp, _c_i32, _c_i32, _c_i32,
                                            _c_i32, _c_i32, _c_i32, _c_i32, ctypes.POINTER(CascadeSizes),
                                            _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_i32,
                                            _c_i32]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _host_i(t, name, dtype):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous host {dtype} tensor")
    return t


def validate_page_table(kv_indptr, kv_indices, kv_lens, num_pages: int, page_size: int,
                        min_len: int = 1) -> None:
    """Check host page-table metadata before it goes to the device; raises PagedKVError naming
    the first bad request (``.bad``)."""
    _host_i(kv_indptr, "kv_indptr", torch.int32)
    _host_i(kv_indices, "kv_indices", torch.int32)
    _host_i(kv_lens, "kv_lens", torch.int32)
    B = kv_lens.numel()
    if kv_indptr.numel() != B + 1:
        raise ValueError("kv_indptr must have batch_size + 1 entries")
    bad = ctypes.c_int32(-1)
    st = load().pkv_validate_page_table(_ptr(kv_indptr), _ptr(kv_indices), _ptr(kv_lens), B,
                                        int(num_pages), int(page_size), int(min_len), ctypes.byref(bad))
    if st != 0:
        e = PagedKVError(f"pkv_validate_page_table (request {bad.value})", st)
        e.bad = bad.value
        raise e


def validate_slots(slot_mapping, num_slots: int) -> None:
    """Check a host slot mapping (in range, no slot twice); raises PagedKVError naming the first
    bad token (``.bad``)."""
    _host_i(slot_mapping, "slot_mapping", torch.int64)
    bad = ctypes.c_int32(-1)
    st = load().pkv_validate_slots(_ptr(slot_mapping), slot_mapping.numel(), int(num_slots),
                                   ctypes.byref(bad))
    if st != 0:
        e = PagedKVError(f"pkv_validate_slots (token {bad.value})", st)
        e.bad = bad.value
        raise e


def selftest_bounded_wait(err_word, stream=None) -> None:
    """Run the bounded-wait check: a GPU wait that nothing completes gives up after its limit and
    ORs DEVERR_TIMEOUT into err_word (int32 [1] on the device)."""
    _need(err_word, "err_word", torch.int32)
    dev = err_word.device
    with torch.cuda.device(dev):
        _call("pkv_selftest_bounded_wait", _ptr(err_word), _stream_ptr(stream, dev))


def status_string(status: int) -> str:
    return load().pkv_status_string(int(status)).decode()


def version() -> int:
    return int(load().pkv_version())


# ---------------------------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------------------------
def _need(t: torch.Tensor, name: str, dtype, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream, device):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _pool(k_pool: torch.Tensor, v_pool: torch.Tensor) -> Pool:
    _need(k_pool, "k_pool", torch.bfloat16)
    _need(v_pool, "v_pool", torch.bfloat16, k_pool.device)
    if k_pool.dim() != 4 or k_pool.shape != v_pool.shape:
        raise ValueError("k_pool and v_pool must both be [num_pages, page_size, num_kv_heads, head_dim]")
    n, ps, hkv, d = k_pool.shape
    return Pool(k_pool.data_ptr(), v_pool.data_ptr(), n, ps, hkv, d)


def _call(fn: str, *args):
    st = getattr(load(), fn)(*args)
    if st != 0:
        raise PagedKVError(fn, st)


# ---------------------------------------------------------------------------------------------
# operations
# ---------------------------------------------------------------------------------------------
def kv_append(k_pool, v_pool, k_new, v_new, slot_mapping, err_word=None, stream=None) -> None:
    """Write k_new[t], v_new[t] into pool slot slot_mapping[t] (negative = skip). In place."""
    pool = _pool(k_pool, v_pool)
    dev = k_pool.device
    _need(k_new, "k_new", torch.bfloat16, dev)
    _need(v_new, "v_new", torch.bfloat16, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, dev)
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, dev)
    T = slot_mapping.numel()
    if k_new.shape != (T, pool.num_kv_heads, pool.head_dim) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [num_tokens, num_kv_heads, head_dim]")
    with torch.cuda.device(dev):
        _call("pkv_kv_append", ctypes.byref(pool), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), T,
              _ptr(err_word), _stream_ptr(stream, dev))


def rope_cos_sin_table(max_position: int, head_dim: int, theta: float, device=None, out=None,
                       stream=None) -> torch.Tensor:
    """The fp32 [max_position, head_dim] cos/sin table rope_kv_append reads (row p: cos of the
    angles p * theta^(-2i/D), then their sines), computed by the library on ``device`` (default:
    the current CUDA device).  Built once, like a model's rotary buffer."""
    dev = torch.device(device) if device is not None else torch.device("cuda")
    if dev.type == "cuda" and dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    if out is None:
        out = torch.empty((max_position, head_dim), dtype=torch.float32, device=dev)
    _need(out, "out", torch.float32, dev)
    if out.shape != (max_position, head_dim):
        raise ValueError("out must be [max_position, head_dim]")
    with torch.cuda.device(dev):
        _call("pkv_rope_cos_sin_table", _ptr(out), int(max_position), int(head_dim), float(theta),
              _stream_ptr(stream, dev))
    return out


def rope_kv_append(k_pool, v_pool, k_new, v_new, slot_mapping, positions, cos_sin, q=None,
                   err_word=None, stream=None) -> None:
    """Rotate k_new (and q in place) by their positions and write K/V into the pool slots."""
    pool = _pool(k_pool, v_pool)
    dev = k_pool.device
    _need(k_new, "k_new", torch.bfloat16, dev)
    _need(v_new, "v_new", torch.bfloat16, dev)
    _need(slot_mapping, "slot_mapping", torch.int64, dev)
    _need(positions, "positions", torch.int32, dev)
    _need(cos_sin, "cos_sin", torch.float32, dev)
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, dev)
    T = slot_mapping.numel()
    if k_new.shape != (T, pool.num_kv_heads, pool.head_dim) or v_new.shape != k_new.shape:
        raise ValueError("k_new/v_new must be [num_tokens, num_kv_heads, head_dim]")
    if positions.numel() != T or cos_sin.dim() != 2 or cos_sin.shape[1] != pool.head_dim:
        raise ValueError("positions must be [num_tokens] and cos_sin [max_position, head_dim]")
    Hq = 0
    if q is not None:
        _need(q, "q", torch.bfloat16, dev)
        if q.dim() != 3 or q.shape[0] != T or q.shape[2] != pool.head_dim:
            raise ValueError("q must be [num_tokens, num_q_heads, head_dim]")
        Hq = q.shape[1]
    with torch.cuda.device(dev):
        _call("pkv_rope_kv_append", ctypes.byref(pool), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping),
              _ptr(positions), _ptr(cos_sin), cos_sin.shape[0], _ptr(q), Hq, T, _ptr(err_word),
              _stream_ptr(stream, dev))


def paged_gather(k_pool, v_pool, kv_indptr, kv_indices, kv_lens, total_len: int, err_word=None,
                 stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Every request's K/V rows in position order, concatenated: [total_len, Hkv, D] each."""
    pool = _pool(k_pool, v_pool)
    dev = k_pool.device
    for t, n in ((kv_indptr, "kv_indptr"), (kv_indices, "kv_indices"), (kv_lens, "kv_lens")):
        _need(t, n, torch.int32, dev)
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, dev)
    B = kv_lens.numel()
    k_out = torch.empty((total_len, pool.num_kv_heads, pool.head_dim), dtype=torch.bfloat16, device=dev)
    v_out = torch.empty_like(k_out)
    with torch.cuda.device(dev):
        _call("pkv_paged_gather", ctypes.byref(pool), _ptr(kv_indptr), _ptr(kv_indices), _ptr(kv_lens),
              B, _ptr(k_out), _ptr(v_out), _ptr(err_word), _stream_ptr(stream, dev))
    return k_out, v_out


def decode_workspace_size(batch_size, num_q_heads, num_kv_heads, head_dim, device=None) -> int:
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        return int(load().pkv_decode_workspace_size(batch_size, num_q_heads, num_kv_heads, head_dim))


def paged_decode(q, k_pool, v_pool, kv_indptr, kv_indices, kv_lens, sm_scale: float, out=None,
                 lse=None, workspace=None, err_word=None, stream=None, return_lse=True, max_ctas=0,
                 l2_keep_tokens=None):
    """Decode attention of q [B, Hq, D] over each request's paged KV. Returns (out, lse).
    ``max_ctas`` > 0 runs it on at most that many SMs (the rest stay free for other streams).
    ``l2_keep_tokens`` (int32 [B] on the device): request b's first l2_keep_tokens[b] positions
    are kept in L2 ahead of the rest (a prefix other requests of the batch share); the results
    do not change."""
    pool = _pool(k_pool, v_pool)
    dev = k_pool.device
    _need(q, "q", torch.bfloat16, dev)
    for t, n in ((kv_indptr, "kv_indptr"), (kv_indices, "kv_indices"), (kv_lens, "kv_lens")):
        _need(t, n, torch.int32, dev)
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, dev)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, dev)
    with torch.cuda.device(dev):
        need = int(load().pkv_decode_workspace_size(B, Hq, pool.num_kv_heads, D))
        if workspace is None:
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        _need(workspace, "workspace", torch.uint8, dev)
        if l2_keep_tokens is not None:
            _need(l2_keep_tokens, "l2_keep_tokens", torch.int32, dev)
            if l2_keep_tokens.shape != (B,):
                raise ValueError("l2_keep_tokens must be [batch_size]")
            _call("pkv_paged_decode_l2keep", ctypes.byref(pool), _ptr(q), B, Hq, _ptr(kv_indptr),
                  _ptr(kv_indices), _ptr(kv_lens), float(sm_scale), _ptr(out), _ptr(lse),
                  _ptr(workspace), workspace.numel(), _ptr(err_word), int(max_ctas),
                  _ptr(l2_keep_tokens), _stream_ptr(stream, dev))
        elif max_ctas:
            _call("pkv_paged_decode_ctas", ctypes.byref(pool), _ptr(q), B, Hq, _ptr(kv_indptr),
                  _ptr(kv_indices), _ptr(kv_lens), float(sm_scale), _ptr(out), _ptr(lse),
                  _ptr(workspace), workspace.numel(), _ptr(err_word), int(max_ctas),
                  _stream_ptr(stream, dev))
        else:
            _call("pkv_paged_decode", ctypes.byref(pool), _ptr(q), B, Hq, _ptr(kv_indptr),
                  _ptr(kv_indices), _ptr(kv_lens), float(sm_scale), _ptr(out), _ptr(lse),
                  _ptr(workspace), workspace.numel(), _ptr(err_word), _stream_ptr(stream, dev))
    return out, lse


def paged_decode_noalloc(q, k_pool, v_pool, kv_indptr, kv_indices, kv_lens, sm_scale: float,
                         out=None, lse=None, err_word=None, stream=None, return_lse=True):
    """paged_decode with the split partials in the library's own device scratch (no workspace
    argument, nothing allocated per call). Returns (out, lse)."""
    pool = _pool(k_pool, v_pool)
    dev = k_pool.device
    _need(q, "q", torch.bfloat16, dev)
    for t, n in ((kv_indptr, "kv_indptr"), (kv_indices, "kv_indices"), (kv_lens, "kv_lens")):
        _need(t, n, torch.int32, dev)
    B, Hq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, dev)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, dev)
    with torch.cuda.device(dev):
        _call("pkv_paged_decode_noalloc", ctypes.byref(pool), _ptr(q), B, Hq, _ptr(kv_indptr),
              _ptr(kv_indices), _ptr(kv_lens), float(sm_scale), _ptr(out), _ptr(lse), _ptr(err_word),
              _stream_ptr(stream, dev))
    return out, lse


def extend_workspace_size(batch_size, num_q_heads, num_kv_heads, head_dim, max_extend_len,
                          device=None) -> int:
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        return int(load().pkv_extend_workspace_size(batch_size, num_q_heads, num_kv_heads, head_dim,
                                                    max_extend_len))


def paged_extend(q, k_pool, v_pool, qo_indptr, kv_indptr, kv_indices, prefix_lens,
                 max_extend_len: int, sm_scale: float, out=None, lse=None, workspace=None,
                 err_word=None, stream=None, return_lse=True):
    """Ragged extend attention with a cached-prefix causal offset. Returns (out, lse)."""
    pool = _pool(k_pool, v_pool)
    dev = k_pool.device
    _need(q, "q", torch.bfloat16, dev)
    for t, n in ((qo_indptr, "qo_indptr"), (kv_indptr, "kv_indptr"), (kv_indices, "kv_indices"),
                 (prefix_lens, "prefix_lens")):
        _need(t, n, torch.int32, dev)
    N, Hq, D = q.shape
    B = prefix_lens.numel()
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, dev)
    if lse is None and return_lse:
        lse = torch.empty((N, Hq), dtype=torch.float32, device=dev)
    if lse is not None:
        _need(lse, "lse", torch.float32, dev)
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, dev)
    with torch.cuda.device(dev):
        need = int(load().pkv_extend_workspace_size(B, Hq, pool.num_kv_heads, D, max_extend_len))
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        if workspace is not None:
            _need(workspace, "workspace", torch.uint8, dev)
        _call("pkv_paged_extend", ctypes.byref(pool), _ptr(q), N, _ptr(qo_indptr), B, Hq, _ptr(kv_indptr),
              _ptr(kv_indices), _ptr(prefix_lens), int(max_extend_len), float(sm_scale), _ptr(out),
              _ptr(lse), _ptr(workspace), 0 if workspace is None else workspace.numel(),
              _ptr(err_word), _stream_ptr(stream, dev))
    return out, lse


def merge_states(o_parts, lse_parts, out=None, lse=None, stream=None):
    """LSE merge of split partials o_parts [S, N, H, D] (fp32 or bf16), lse_parts [S, N, H] fp32."""
    dev = o_parts.device
    bf16 = o_parts.dtype == torch.bfloat16
    fn = "pkv_merge_states_bf16" if bf16 else "pkv_merge_states"
    _need(o_parts, "o_parts", torch.bfloat16 if bf16 else torch.float32)
    _need(lse_parts, "lse_parts", torch.float32, dev)
    S, N, H, D = o_parts.shape
    if lse_parts.shape != (S, N, H):
        raise ValueError("lse_parts must be [S, N, H]")
    if out is None:
        out = torch.empty((N, H, D), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((N, H), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, dev)
    _need(lse, "lse", torch.float32, dev)
    with torch.cuda.device(dev):
        _call(fn, _ptr(o_parts), _ptr(lse_parts), S, N, H, D, _ptr(out), _ptr(lse),
              _stream_ptr(stream, dev))
    return out, lse


def shared_prefix_workspace_size(num_parts, num_q_heads, num_kv_heads, head_dim, max_part_rows,
                                 device=None) -> int:
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        return int(load().pkv_shared_prefix_workspace_size(num_parts, num_q_heads, num_kv_heads,
                                                           head_dim, max_part_rows))


def shared_prefix_attention(q, k_pool, v_pool, q_start, q_len, o_start, kv_indptr, kv_indices,
                            kv_lens, max_part_rows: int, sm_scale: float, o_part, lse_part=None,
                            workspace=None, err_word=None, stream=None):
    """Unmasked attention of each part's query rows over the part's (shared) pages: the partial
    states of a cascade level, written at rows o_start[p].. of o_part (bf16) and lse_part."""
    pool = _pool(k_pool, v_pool)
    dev = k_pool.device
    _need(q, "q", torch.bfloat16, dev)
    for t, n in ((q_start, "q_start"), (q_len, "q_len"), (o_start, "o_start"), (kv_indptr, "kv_indptr"),
                 (kv_indices, "kv_indices"), (kv_lens, "kv_lens")):
        _need(t, n, torch.int32, dev)
    _need(o_part, "o_part", torch.bfloat16, dev)
    Nq, Hq, D = q.shape
    if o_part.dim() != 3 or o_part.shape[1:] != q.shape[1:]:
        raise ValueError("o_part must be [num_out_rows, num_q_heads, head_dim]")
    n_out = o_part.shape[0]
    if lse_part is not None:
        _need(lse_part, "lse_part", torch.float32, dev)
        if lse_part.shape != (n_out, Hq):
            raise ValueError("lse_part must be [num_out_rows, num_q_heads]")
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, dev)
    P = kv_lens.numel()
    with torch.cuda.device(dev):
        need = int(load().pkv_shared_prefix_workspace_size(P, Hq, pool.num_kv_heads, D, max_part_rows))
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        if workspace is not None:
            _need(workspace, "workspace", torch.uint8, dev)
        _call("pkv_shared_prefix_attention", ctypes.byref(pool), _ptr(q), Nq, _ptr(q_start), _ptr(q_len),
              _ptr(o_start), P, Hq, _ptr(kv_indptr), _ptr(kv_indices), _ptr(kv_lens), int(max_part_rows),
              float(sm_scale), _ptr(o_part), _ptr(lse_part), n_out, _ptr(workspace),
              0 if workspace is None else workspace.numel(), _ptr(err_word), _stream_ptr(stream, dev))
    return o_part, lse_part


def cascade_decode(q, k_pool, v_pool, plan, sm_scale: float, out=None, lse=None, o_parts=None,
                   lse_parts=None, prefix_workspace=None, decode_workspace=None, err_word=None,
                   stream=None):
    """Decode through a shared-prefix plan (``cascade.plan_shared_prefix``, its tensors on the
    device): the shared-prefix states, the decode over each request's own pages into the last
    split, and their log-sum-exp merge.  Three library calls on one stream; returns (out, lse)."""
    dev = q.device
    B, Hq, D = q.shape
    S = plan.num_splits
    if o_parts is None:
        o_parts = torch.empty((S + 1, B, Hq, D), dtype=torch.bfloat16, device=dev)
    if lse_parts is None:
        lse_parts = torch.empty((S + 1, B, Hq), dtype=torch.float32, device=dev)
    if o_parts.shape != (S + 1, B, Hq, D) or lse_parts.shape != (S + 1, B, Hq):
        raise ValueError("o_parts / lse_parts must be [num_splits + 1, B, Hq, (D)]")
    shared_prefix_attention(q, k_pool, v_pool, plan.part_q_start, plan.part_q_len, plan.part_o_start,
                            plan.part_kv_indptr, plan.part_kv_indices, plan.part_kv_lens,
                            plan.max_part_rows, sm_scale, o_parts.view(-1, Hq, D),
                            lse_parts.view(-1, Hq), workspace=prefix_workspace, err_word=err_word,
                            stream=stream)
    paged_decode(q, k_pool, v_pool, plan.suffix_kv_indptr, plan.suffix_kv_indices, plan.suffix_kv_lens,
                 sm_scale, out=o_parts[S], lse=lse_parts[S], workspace=decode_workspace,
                 err_word=err_word, stream=stream)
    return merge_states(o_parts, lse_parts, out=out, lse=lse, stream=stream)
