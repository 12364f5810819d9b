"""Fused RoPE + KV append on the GPU against the fp64 oracle.

Tolerance from the arithmetic: the kernel forms x_i cos - x_j sin in fp32 (two products and an FMA,
each within 2^-24 relative) from a cos/sin table rounded to fp32, then rounds to bf16 (within half
an ulp; bf16 has 8 significand bits, so half an ulp is at most 2^-8 of the value).  So
|gpu - exact| <= 2^-8 |exact| + 2^-21 (|x_i| + |x_j|) element-wise.
V rows are copied and must be bit-exact; every other pool slot must be left unchanged."""

import numpy as np
import pytest
import torch

import oracle
from workloads import random_small_batch
from _gpu_helpers import DeviceBatch, assert_attention_close, bits_equal

pytestmark = pytest.mark.gpu

THETA = 1.0e6  # Qwen3's rotary base


def _bound_ok(gpu_bf16, exact, x):
    D = exact.shape[-1]
    g = gpu_bf16.float().cpu().numpy().astype(np.float64)
    pair = np.abs(x[..., : D // 2]) + np.abs(x[..., D // 2:])
    pair = np.concatenate([pair, pair], axis=-1)
    tol = 2.0 ** -8 * np.abs(exact) + 2.0 ** -21 * pair
    return np.all(np.abs(g - exact) <= tol), float(np.max(np.abs(g - exact) - tol))


def _positions(b, gen):
    return torch.randint(0, 32768, (b.num_new_tokens,), generator=gen, dtype=torch.int32)


@pytest.mark.parametrize("npos,D,theta", [(100, 128, THETA), (32768, 128, THETA), (4096, 64, 1.0e4)])
def test_table_matches_oracle_angles(lib, npos, D, theta):
    # the library builds the table on the device from double-precision angles; each entry is
    # within an fp32 rounding (2^-25 of a value at most 1) of the fp64 cos/sin
    t = lib.rope_cos_sin_table(npos, D, theta).cpu()
    ang = oracle.rope_angles(np.arange(npos), D, theta)
    assert np.abs(t[:, : D // 2].double().numpy() - np.cos(ang)).max() < 1e-7
    assert np.abs(t[:, D // 2:].double().numpy() - np.sin(ang)).max() < 1e-7


@pytest.mark.parametrize("hkv,hq,D", [(8, 32, 128), (2, 14, 64)])
def test_rope_append_against_oracle(lib, hkv, hq, D):
    b = random_small_batch(71 + D, page_size=16, num_q_heads=hq, num_kv_heads=hkv, head_dim=D,
                           decode_lens=(40, 900, 3), decode_new=2, extend=((100, 250), (0, 33)))
    gen = torch.Generator().manual_seed(5)
    pos = _positions(b, gen)
    slots = b.slot_mapping.clone()
    slots[3] = -1  # padding token
    q = torch.randn((b.num_new_tokens, hq, D), generator=gen).to(torch.bfloat16)
    d = DeviceBatch(b)
    qd = q.cuda()
    table = lib.rope_cos_sin_table(32768, D, THETA, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.rope_kv_append(d.k_pool, d.v_pool, d.k_new, d.v_new, slots.cuda(), pos.cuda(), table, q=qd,
                       err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kp_ref, vp_ref, k_rot = oracle.rope_kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, slots, pos, 16, THETA)
    assert bits_equal(d.v_pool, vp_ref)
    written = slots >= 0
    s_ok = slots[written]
    got = d.k_pool.cpu().view(-1, hkv, D)[s_ok]
    ok, worst = _bound_ok(got, k_rot[written.numpy()], oracle.as_f64(b.k_new)[written.numpy()])
    assert ok, worst
    # slots outside the step are untouched
    mask = torch.ones(b.num_pages * 16, dtype=torch.bool)
    mask[s_ok] = False
    assert bits_equal(d.k_pool.cpu().view(-1, hkv, D)[mask], b.k_pool.view(-1, hkv, D)[mask])
    q_rot = oracle.rope(oracle.as_f64(q), pos, THETA)
    ok, worst = _bound_ok(qd, q_rot, oracle.as_f64(q))
    assert ok, worst


def test_rope_append_reports_bad_position(lib):
    b = random_small_batch(81, page_size=16, num_q_heads=8, num_kv_heads=2, head_dim=64, decode_lens=(20,))
    d = DeviceBatch(b)
    pos = torch.tensor([70000], dtype=torch.int32)
    table = lib.rope_cos_sin_table(1024, 64, THETA, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.rope_kv_append(d.k_pool, d.v_pool, d.k_new, d.v_new, d.slot_mapping, pos.cuda(), table, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & lib.DEVERR_LENGTH
    assert bits_equal(d.k_pool, b.k_pool)  # nothing written


def test_rope_append_then_decode(lib):
    """The fused step before attention: rotate q and new k, append, decode; against the oracle
    doing the same (its own bf16 rounding of the fp64 rotation)."""
    b = random_small_batch(91, page_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128,
                           decode_lens=(17, 600, 2500), decode_new=1)
    pos = (b.dec_kv_lens - 1).to(torch.int32)  # the new token sits at the last position
    d = DeviceBatch(b)
    table = lib.rope_cos_sin_table(4096, 128, THETA, device="cuda")
    lib.rope_kv_append(d.k_pool, d.v_pool, d.k_new, d.v_new, d.slot_mapping, pos.cuda(), table, q=d.dec_q)
    out, lse = lib.paged_decode(d.dec_q, d.k_pool, d.v_pool, d.dec_kv_indptr, d.dec_kv_indices,
                                d.dec_kv_lens, b.sm_scale)
    kp, vp, _ = oracle.rope_kv_append(b.k_pool, b.v_pool, b.k_new, b.v_new, b.slot_mapping, pos, 16, THETA)
    q_rot = torch.tensor(oracle.rope(oracle.as_f64(b.dec_q), pos, THETA)).to(torch.bfloat16)
    o_ref, l_ref = oracle.paged_decode(q_rot, kp, vp, b.dec_kv_indptr, b.dec_kv_indices, b.dec_kv_lens,
                                       16, b.sm_scale)
    assert_attention_close(out, lse, o_ref, l_ref, what="rope + decode")
