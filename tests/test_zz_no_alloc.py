"""The no-allocation decode entry point, called through the C ABI.

pkv_paged_decode_noalloc serves callers that cannot allocate device memory when they decode (an
engine whose KV pool was given a fixed share of HBM up front, or code that must not take
cudaMalloc's implicit synchronisation mid-step): it keeps its split partials in a scratch array the
library holds in device memory.  Its results must equal those of pkv_paged_decode with a
caller-supplied workspace and the fp64 oracle's, on consecutive calls that reuse the same scratch.

This file is named to be collected last, so a run that stops at the first failure has already run
every other test; it also passes on its own in a fresh process.
"""

import ctypes
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import random_small_batch
from _gpu_helpers import O_MAX_ABS, O_MEAN_ABS, LSE_ABS

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SCRATCH_BYTES = 16 * 1024 * 1024  # PKV_DECODE_NOALLOC_SCRATCH_BYTES


class Pool(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("num_pages", ctypes.c_int64),
                ("page_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32)]


@pytest.fixture(scope="module")
def cdll():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_attention_10_gb300 import build

    lib = ctypes.CDLL(build.build())
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    P = ctypes.POINTER(Pool)
    lib.pkv_paged_decode.restype = i32
    lib.pkv_paged_decode.argtypes = [P, vp, i32, i32, vp, vp, vp, f32, vp, vp, vp, sz, vp, vp]
    lib.pkv_paged_decode_noalloc.restype = i32
    lib.pkv_paged_decode_noalloc.argtypes = [P, vp, i32, i32, vp, vp, vp, f32, vp, vp, vp, vp]
    lib.pkv_decode_workspace_size.restype = sz
    lib.pkv_decode_workspace_size.argtypes = [i32, i32, i32, i32]
    return lib


def _device_batch(seed, lens, hq=32, hkv=8, D=128, ps=16):
    b = random_small_batch(seed, page_size=ps, num_q_heads=hq, num_kv_heads=hkv, head_dim=D,
                           decode_lens=lens, decode_new=1)
    kp, vp = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, ps)
    t = dict(kp=kp.cuda(), vp=vp.cuda(), q=b.dec_q.cuda(), ind=b.dec_kv_indptr.cuda(),
             idx=b.dec_kv_indices.cuda(), lens=b.dec_kv_lens.cuda())
    pool = Pool(t["kp"].data_ptr(), t["vp"].data_ptr(), b.num_pages, ps, hkv, D)
    return b, t, pool


def _p(x):
    return ctypes.c_void_p(x.data_ptr())


def _decode_pair(cdll, b, t, pool):
    """(out, lse) from the workspace entry point and from the no-alloc entry point, and the two
    calls' device error words (both start at zero)."""
    B, hq = b.num_decode, b.num_q_heads
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ws_bytes = cdll.pkv_decode_workspace_size(B, hq, b.num_kv_heads, b.head_dim)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    err = torch.zeros(2, dtype=torch.int32, device="cuda")
    out_ref = torch.empty_like(t["q"])
    lse_ref = torch.empty((B, hq), dtype=torch.float32, device="cuda")
    st = cdll.pkv_paged_decode(ctypes.byref(pool), _p(t["q"]), B, hq, _p(t["ind"]), _p(t["idx"]),
                               _p(t["lens"]), b.sm_scale, _p(out_ref), _p(lse_ref), _p(ws), ws_bytes,
                               _p(err[0:1]), stream)
    assert st == 0
    out = torch.full_like(t["q"], float("nan"))
    lse = torch.full((B, hq), float("nan"), dtype=torch.float32, device="cuda")
    st = cdll.pkv_paged_decode_noalloc(ctypes.byref(pool), _p(t["q"]), B, hq, _p(t["ind"]),
                                       _p(t["idx"]), _p(t["lens"]), b.sm_scale, _p(out), _p(lse),
                                       _p(err[1:2]), stream)
    assert st == 0
    torch.cuda.synchronize()
    return out_ref, lse_ref, out, lse, err.cpu().tolist()


def test_noalloc_decode_matches_workspace_decode_twice(cdll):
    # two calls in a row: long split requests first, then a different batch that reuses the
    # scratch the first call left behind.  Each is checked against the workspace decode and
    # against the fp64 oracle, and neither call may raise a device error bit (a merge that read a
    # stale entry of the reused scratch would show up in the output or in the error word).
    for seed, lens in ((41, (3000, 17, 9000, 1, 640, 2049)), (42, (5, 700, 33, 4096, 128))):
        b, t, pool = _device_batch(seed, lens)
        out_ref, lse_ref, out, lse, err = _decode_pair(cdll, b, t, pool)
        assert err == [0, 0]
        d = (out.float() - out_ref.float()).abs()
        assert d.max().item() <= O_MAX_ABS and d.mean().item() <= O_MEAN_ABS
        assert (lse - lse_ref).abs().max().item() <= LSE_ABS
        kp, vp = t["kp"].cpu(), t["vp"].cpu()
        o_or, lse_or = oracle.paged_decode(b.dec_q, kp, vp, b.dec_kv_indptr, b.dec_kv_indices,
                                           b.dec_kv_lens, b.page_size, b.sm_scale)
        do = np.abs(out.float().cpu().numpy().astype(np.float64) - o_or)
        assert do.max() <= O_MAX_ABS and do.mean() <= O_MEAN_ABS, (do.max(), do.mean())
        assert np.abs(lse.cpu().numpy().astype(np.float64) - lse_or).max() <= LSE_ABS


def test_noalloc_rejects_shapes_beyond_its_scratch(cdll):
    # a batch whose split partials need more than the fixed scratch is refused on the host
    B, hq, hkv, D = 4000, 64, 8, 128
    need = cdll.pkv_decode_workspace_size(B, hq, hkv, D)
    assert need > SCRATCH_BYTES
    dummy = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    pool = Pool(dummy.data_ptr(), dummy.data_ptr(), 1, 16, hkv, D)
    st = cdll.pkv_paged_decode_noalloc(ctypes.byref(pool), _p(dummy), B, hq, _p(dummy), _p(dummy),
                                       _p(dummy), 1.0, _p(dummy), None, None, None)
    assert st == 3  # PKV_ERR_WORKSPACE, nothing launched


def test_noalloc_binding_matches_paged_decode(lib):
    # the same entry point through the Python binding, against the workspace decode
    b, t, pool = _device_batch(43, (1500, 64, 777))
    out_ref, lse_ref = lib.paged_decode(t["q"], t["kp"], t["vp"], t["ind"], t["idx"], t["lens"],
                                        b.sm_scale)
    out, lse = lib.paged_decode_noalloc(t["q"], t["kp"], t["vp"], t["ind"], t["idx"], t["lens"],
                                        b.sm_scale)
    torch.cuda.synchronize()
    d = (out.float() - out_ref.float()).abs()
    assert d.max().item() <= O_MAX_ABS and d.mean().item() <= O_MEAN_ABS
    assert (lse - lse_ref).abs().max().item() <= LSE_ABS
