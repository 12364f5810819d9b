"""The shared-prefix (cascade) decode and the fused RoPE append driven through the C ABI alone.

A C caller plans the cascade with pkv_plan_shared_prefix on host copies of its page lists, copies
the plan to the device and runs pkv_shared_prefix_attention, pkv_paged_decode (each request's own
pages, into the last split) and pkv_merge_states_bf16; for the RoPE append it builds the cos/sin
table with pkv_rope_cos_sin_table and calls pkv_rope_kv_append.  Here ctypes stands in for that
caller: torch only allocates device memory and copies bytes, and every step of the path runs in
the library.  Results are checked against the fp64 oracle.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from workloads import random_small_batch
from _gpu_helpers import assert_attention_close, bits_equal

pytestmark = pytest.mark.gpu

vp, i32, f32, sz, f64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t, ctypes.c_double


class Pool(ctypes.Structure):
    _fields_ = [("k", vp), ("v", vp), ("num_pages", ctypes.c_int64), ("page_size", i32),
                ("num_kv_heads", i32), ("head_dim", i32)]


class Sizes(ctypes.Structure):
    _fields_ = [("num_splits", i32), ("num_parts", i32), ("max_part_rows", i32),
                ("num_part_indices", i32), ("num_suffix_indices", i32)]


@pytest.fixture(scope="module")
def cdll():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_attention_10_gb300 import build

    lib = ctypes.CDLL(build.build())
    P = ctypes.POINTER(Pool)
    sigs = {
        "pkv_plan_shared_prefix": [vp, vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                   ctypes.POINTER(Sizes)] + [vp] * 10 + [i32, i32],
        "pkv_shared_prefix_workspace_size": [i32, i32, i32, i32, i32],
        "pkv_shared_prefix_attention": [P, vp, i32, vp, vp, vp, i32, i32, vp, vp, vp, i32, f32, vp, vp,
                                        i32, vp, sz, vp, vp],
        "pkv_decode_workspace_size": [i32, i32, i32, i32],
        "pkv_paged_decode": [P, vp, i32, i32, vp, vp, vp, f32, vp, vp, vp, sz, vp, vp],
        "pkv_merge_states_bf16": [vp, vp, i32, i32, i32, i32, vp, vp, vp],
        "pkv_rope_cos_sin_table": [vp, i32, i32, f64, vp],
        "pkv_rope_kv_append": [P, vp, vp, vp, vp, vp, i32, vp, i32, i32, vp, vp],
    }
    for name, args in sigs.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = sz if name.endswith("workspace_size") else i32
    return lib


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_cascade_decode_through_the_c_abi(cdll):
    ps, Hq, Hkv, D = 16, 32, 8, 128
    b = random_small_batch(77, page_size=ps, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                           decode_lens=(40, 700, 900, 1300, 650, 90), decode_new=1, share_decode_prefix=512)
    sharers = [i for i, r in enumerate(b.requests) if r.share_group == 0]
    assert len(sharers) >= 3 and sharers == list(range(sharers[0], sharers[0] + len(sharers)))
    kp, vpool = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, ps)
    B = b.num_decode
    # host plan: a size query, then the arrays
    ind, idx, lens = b.dec_kv_indptr.contiguous(), b.dec_kv_indices.contiguous(), b.dec_kv_lens.contiguous()
    gf = torch.tensor([sharers[0]], dtype=torch.int32)
    gc = torch.tensor([len(sharers)], dtype=torch.int32)
    sizes = Sizes()
    head = (_p(ind), _p(idx), _p(lens), B, _p(gf), _p(gc), 1, ps, Hkv, Hq // Hkv, 152, 2, 128,
            ctypes.byref(sizes))
    assert cdll.pkv_plan_shared_prefix(*head, *([None] * 10), 0, 0) == 0
    S, n_parts = sizes.num_splits, sizes.num_parts
    cap = int(ind[-1])
    host = {k: torch.zeros(n, dtype=torch.int32) for k, n in (
        ("shared", 1), ("q_start", n_parts), ("q_len", n_parts), ("o_start", n_parts),
        ("p_indptr", n_parts + 1), ("p_indices", cap), ("p_lens", n_parts), ("s_indptr", B + 1),
        ("s_indices", cap), ("s_lens", B))}
    order = ("shared", "q_start", "q_len", "o_start", "p_indptr", "p_indices", "p_lens", "s_indptr",
             "s_indices", "s_lens")
    assert cdll.pkv_plan_shared_prefix(*head, *[_p(host[k]) for k in order], n_parts, cap) == 0
    assert int(host["shared"][0]) == 512
    dev = {k: v.cuda() for k, v in host.items()}
    q, kpd, vpd = b.dec_q.cuda(), kp.cuda(), vpool.cuda()
    pool = Pool(kpd.data_ptr(), vpd.data_ptr(), b.num_pages, ps, Hkv, D)
    o_parts = torch.empty((S + 1, B, Hq, D), dtype=torch.bfloat16, device="cuda")
    lse_parts = torch.empty((S + 1, B, Hq), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws1 = cdll.pkv_shared_prefix_workspace_size(n_parts, Hq, Hkv, D, sizes.max_part_rows)
    w1 = torch.empty(max(ws1, 16), dtype=torch.uint8, device="cuda")
    st = cdll.pkv_shared_prefix_attention(
        ctypes.byref(pool), _p(q), B, _p(dev["q_start"]), _p(dev["q_len"]), _p(dev["o_start"]), n_parts, Hq,
        _p(dev["p_indptr"]), _p(dev["p_indices"]), _p(dev["p_lens"]), sizes.max_part_rows, b.sm_scale,
        _p(o_parts), _p(lse_parts), S * B, _p(w1), ws1, _p(err), _stream())
    assert st == 0
    ws2 = cdll.pkv_decode_workspace_size(B, Hq, Hkv, D)
    w2 = torch.empty(ws2, dtype=torch.uint8, device="cuda")
    st = cdll.pkv_paged_decode(ctypes.byref(pool), _p(q), B, Hq, _p(dev["s_indptr"]), _p(dev["s_indices"]),
                               _p(dev["s_lens"]), b.sm_scale, _p(o_parts[S]), _p(lse_parts[S]), _p(w2), ws2,
                               _p(err), _stream())
    assert st == 0
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    st = cdll.pkv_merge_states_bf16(_p(o_parts), _p(lse_parts), S + 1, B, Hq, D, _p(out), _p(lse), _stream())
    assert st == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o_ref, lse_ref = oracle.paged_decode(b.dec_q, kp, vpool, b.dec_kv_indptr, b.dec_kv_indices,
                                         b.dec_kv_lens, ps, b.sm_scale)
    assert_attention_close(out, lse, o_ref, lse_ref, what="cascade through the C ABI")


def test_rope_append_through_the_c_abi(cdll):
    ps, Hq, Hkv, D, theta = 16, 32, 8, 128, 1.0e6
    b = random_small_batch(78, page_size=ps, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                           decode_lens=(40, 900, 3), decode_new=2, extend=((100, 250),))
    gen = torch.Generator().manual_seed(9)
    T = b.num_new_tokens
    pos = torch.randint(0, 8192, (T,), generator=gen, dtype=torch.int32)
    max_pos = 8192
    table = torch.empty((max_pos, D), dtype=torch.float32, device="cuda")
    assert cdll.pkv_rope_cos_sin_table(_p(table), max_pos, D, theta, _stream()) == 0
    kpd, vpd = b.k_pool.cuda(), b.v_pool.cuda()
    pool = Pool(kpd.data_ptr(), vpd.data_ptr(), b.num_pages, ps, Hkv, D)
    kn, vn, sl, pd = b.k_new.cuda(), b.v_new.cuda(), b.slot_mapping.cuda(), pos.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = cdll.pkv_rope_kv_append(ctypes.byref(pool), _p(kn), _p(vn), _p(sl), _p(pd), _p(table), max_pos,
                                 None, 0, T, _p(err), _stream())
    assert st == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kp_ref, vp_ref, k_rot = oracle.rope_kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping,
                                                  pos, ps, theta)
    assert bits_equal(vpd, vp_ref)
    # K: within the fp32 rotation's rounding plus one bf16 rounding of the fp64 value
    got = kpd.view(-1, Hkv, D)[b.slot_mapping.cuda()].float().cpu().numpy().astype(np.float64)
    x = np.abs(b.k_new.double().numpy())
    pair = np.concatenate([x[..., : D // 2] + x[..., D // 2:]] * 2, axis=-1)
    assert (np.abs(got - k_rot) <= 2.0 ** -8 * np.abs(k_rot) + 2.0 ** -21 * pair).all()
    # every slot the append does not own is unchanged
    keep = torch.ones(kpd.view(-1, Hkv, D).shape[0], dtype=torch.bool)
    keep[b.slot_mapping] = False
    assert bits_equal(kpd.view(-1, Hkv, D).cpu()[keep], b.k_pool.view(-1, Hkv, D)[keep])


def test_l2keep_decode_through_the_c_abi(cdll):
    """pkv_paged_decode_l2keep called as a C caller would: with each request's shared length it
    returns exactly what pkv_paged_decode returns (the hint steers L2 evictions only)."""
    ps, Hq, Hkv, D = 16, 32, 8, 128
    b = random_small_batch(79, page_size=ps, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                           decode_lens=(40, 700, 900, 1300), decode_new=1, share_decode_prefix=256)
    kp, vpool = oracle.kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, ps)
    f = cdll.pkv_paged_decode_l2keep
    f.argtypes = [ctypes.POINTER(Pool), vp, i32, i32, vp, vp, vp, f32, vp, vp, vp, sz, vp, i32, vp, vp]
    f.restype = i32
    B = b.num_decode
    q, kpd, vpd = b.dec_q.cuda(), kp.cuda(), vpool.cuda()
    pool = Pool(kpd.data_ptr(), vpd.data_ptr(), b.num_pages, ps, Hkv, D)
    ind, idx, lens = b.dec_kv_indptr.cuda(), b.dec_kv_indices.cuda(), b.dec_kv_lens.cuda()
    keep = b.dec_shared_tokens.cuda()
    ws = cdll.pkv_decode_workspace_size(B, Hq, Hkv, D)
    w = torch.empty(ws, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for hinted in (True, False):
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
        if hinted:
            st = f(ctypes.byref(pool), _p(q), B, Hq, _p(ind), _p(idx), _p(lens), b.sm_scale, _p(out), _p(lse),
                   _p(w), ws, _p(err), 0, _p(keep), _stream())
        else:
            st = cdll.pkv_paged_decode(ctypes.byref(pool), _p(q), B, Hq, _p(ind), _p(idx), _p(lens), b.sm_scale,
                                       _p(out), _p(lse), _p(w), ws, _p(err), _stream())
        assert st == 0
        outs.append((out, lse))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1], outs[1][1])
